// K2: the KQ-mask builder.
//
// "llama.cpp and the ubatch", "The mask is doing the work": row i sees cell j
// iff the cell is occupied, holds seq_id[i][0], (causal) pos_j <= pos_i, and
// (sliding window of n_swa positions) pos_i - pos_j < n_swa; everything else is
// -inf before the softmax.  The mask is built on the
// device from the cell mirror (position, sequence bitset, and the serial of
// the ubatch that reserved the cell), once per ubatch, and reused by every
// layer.  Two products:
//   * the attention plan -- for every block of rows (rows sharing a stream and
//     a first sequence id) and every 64-cell tile: how many (row, cell) pairs
//     are visible and which 8-cell groups hold one; then each block's list of
//     tiles with anything visible, and the split-K work items over those
//     lists.  Attention reads K/V only for listed tiles and skips the per-cell
//     test on tiles that are fully visible.
//   * on request, the dense additive F16 mask [n_tokens][n_kv]: 0x0000
//     visible, 0xFC00 (-inf) masked, column j = cell j of the row's stream.

#include "dev_common.cuh"
#include "kernels.h"

namespace {

using kvi::TILE;
using kvi::SUB;

// Rows of block b that see a cell at position cpos (sequence and epoch
// already checked).  The row positions that see it form one interval (from
// cpos under causal attention, to cpos + n_swa - 1 under a window), so the
// block's rows (positions pos_min .. pos_max) all see it when both ends do, and
// none does when the interval misses that range.
__device__ __forceinline__ int32_t rows_seeing(const kvk::UbView &u, const kvi::DevBlock &b,
                                               int32_t cpos) {
    if (kvd::pos_visible(u.causal, u.n_swa, b.pos_min, cpos) && kvd::pos_visible(u.causal, u.n_swa, b.pos_max, cpos))
        return b.n_rows;
    if ((u.causal && cpos > b.pos_max) || (u.n_swa > 0 && (int64_t)b.pos_min - cpos >= u.n_swa)) return 0;
    if (b.contig) {
        // the seeing positions cpos .. cpos + n_swa - 1 (each end open without causality
        // or window) against the block's pos_min .. pos_max, each held by one row
        const int64_t lo = u.causal ? max((int64_t)b.pos_min, (int64_t)cpos) : (int64_t)b.pos_min;
        const int64_t hi = u.n_swa > 0 ? min((int64_t)b.pos_max, (int64_t)cpos + u.n_swa - 1) : (int64_t)b.pos_max;
        return hi >= lo ? (int32_t)(hi - lo + 1) : 0;
    }
    int32_t n = 0;
    for (int32_t k = 0; k < b.n_rows; ++k)
        n += kvd::pos_visible(u.causal, u.n_swa, u.rows[u.perm[b.row0 + k]].pos, cpos) ? 1 : 0;
    return n;
}

// One CTA per (64-cell tile, stream).  Shared counters per block, then one
// plain store per (block of this stream, tile): no global atomics and no
// separate clearing pass.
__global__ void __launch_bounds__(TILE) k_plan_tiles(kvk::UbView u, kvk::Plan p) {
    extern __shared__ uint32_t sh[];
    uint32_t *cnt = sh;                 // [n_blocks]
    uint32_t *sub = sh + u.n_blocks;    // [n_blocks]
    const int32_t t = blockIdx.x;
    const int32_t s = blockIdx.y;
    for (int32_t b = threadIdx.x; b < u.n_blocks; b += blockDim.x) { cnt[b] = 0; sub[b] = 0; }
    __syncthreads();
    const int32_t j = t * TILE + threadIdx.x;
    if (j < u.n_kv) {
        const int64_t g = (int64_t)s * u.kv_size + j;
        if (u.cell_epoch[g] <= u.ub_epoch) {
            const int32_t cpos = u.cell_pos[g];
            for (int32_t w = 0; w < u.n_words; ++w) {
                uint64_t bits = u.cell_bits[g * u.n_words + w];
                while (bits) {
                    const int32_t q = w * 64 + __ffsll((long long)bits) - 1;
                    bits &= bits - 1;
                    for (int32_t k = u.seq_blk_off[q]; k < u.seq_blk_off[q + 1]; ++k) {
                        const int32_t bi = u.seq_blk[k];
                        const int32_t n = rows_seeing(u, u.blocks[bi], cpos);
                        if (n) {
                            atomicAdd(&cnt[bi], (uint32_t)n);
                            atomicOr(&sub[bi], 1u << (threadIdx.x / SUB));
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    for (int32_t b = threadIdx.x; b < u.n_blocks; b += blockDim.x) {
        if (u.blocks[b].stream == s)
            p.flags[(int64_t)b * p.tile_stride + t] = cnt[b] | (sub[b] << 16);
    }
}

// One CTA per block: ordered list of the tiles with any visible pair, and the
// decode cost of the list up to each entry, so that decode work is cut by cost, not
// by tile count.  A fully visible tile costs 8 (its eight 8-cell groups); another
// costs 2 plus the number of its 8-cell groups holding a visible pair (the decode
// kernel loads exactly those groups, and the 2 stands for the per-tile work that
// does not shrink with them: the flag read, the group queueing, the mask).
__global__ void __launch_bounds__(256) k_plan_compact(kvk::UbView u, kvk::Plan p, int32_t n_tiles) {
    __shared__ int32_t warp_sum[8], warp_cost[8];
    __shared__ int32_t base, cbase;
    const int32_t b = blockIdx.x;
    const uint32_t *f = p.flags + (int64_t)b * p.tile_stride;
    int32_t *out = p.tiles + (int64_t)b * p.tile_stride;
    int32_t *cum = p.cum + (int64_t)b * p.tile_stride;
    const int32_t full_cnt = u.blocks[b].n_rows * TILE;
    if (threadIdx.x == 0) {
        base = 0;
        cbase = 0;
    }
    __syncthreads();
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int32_t a = 0; a < n_tiles; a += blockDim.x) {
        const int32_t t = a + threadIdx.x;
        const uint32_t fl = t < n_tiles ? f[t] : 0u;
        const bool nz = fl != 0;
        const int32_t cost = !nz ? 0 : (int32_t)(fl & 0xffffu) == full_cnt ? 8 : 2 + __popc((fl >> 16) & 0xffu);
        const uint32_t bal = __ballot_sync(0xffffffffu, nz);
        const int32_t before = __popc(bal & ((1u << lane) - 1u));
        int32_t incl = cost;   // inclusive warp scan of the costs
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 0) warp_sum[warp] = __popc(bal);
        if (lane == 31) warp_cost[warp] = incl;
        __syncthreads();
        int32_t off = base, coff = cbase;
        for (int32_t w = 0; w < warp; ++w) {
            off += warp_sum[w];
            coff += warp_cost[w];
        }
        if (nz) {
            out[off + before] = t;
            cum[off + before] = coff + incl - cost;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t tot = 0, ctot = 0;
            for (int32_t w = 0; w < (int32_t)(blockDim.x >> 5); ++w) {
                tot += warp_sum[w];
                ctot += warp_cost[w];
            }
            base += tot;
            cbase += ctot;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        p.counts[b] = base;
        p.wcount[b] = cbase;
    }
}

// Decode: the first list entry whose cost-before is at least x (0 .. count).
__device__ __forceinline__ int32_t tile_at_cost(const kvk::Plan &p, int32_t b, int64_t x) {
    const int32_t *cum = p.cum + (int64_t)b * p.tile_stride;
    int32_t lo = 0, hi = p.counts[b];
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (cum[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// One CTA: cut the tile lists into split-K work items.  Per path (decode blocks
// first, then prefill blocks) the CTA columns of the attention grid are filled
// greedily in block order: a column takes the rest of the current block if it
// fits under a budget T, else as much of it as fits, and the block spills into
// the next column.  Every item costs a start-up and an epilogue on top of its
// work, so a column's cost is its work plus a fixed cost per item; T is the
// smallest budget with which the fill needs at most gx columns.  So the columns
// carry about the same time, a block's items are consecutive, and a column takes
// a second block only where the blocks are small next to the budget.  A block
// with an empty list gets one empty item (its rows see nothing and get zeros);
// columns beyond the fill get no item.

// Decode, in the units of the tile costs (a fully visible tile 8): start-up (the
// first stage's latency, the Q load) plus epilogue (the merge of the eight warps'
// states, the partial and its completion count) of one item.
constexpr int64_t DEC_ITEM_COST = 16;
// Decode: no piece smaller than one fully visible tile, unless it ends a block.
constexpr int64_t DEC_MIN_TAKE = 8;
// Decode block costs staged in shared memory for the budget search.
constexpr int32_t DEC_STAGE = 2048;
// Prefill, in units of one step (a pair of 64-cell tiles for both MMA tiles of a
// block): start-up plus epilogue of one item.
constexpr int64_t PF_ITEM_COST = 3;
// Extra cost of the piece that holds a block's last pair (its causal diagonal, with
// the per-cell mask), in the same units.
constexpr int64_t PF_DIAG_COST = 1;
// Extra cost of every piece of a block split over several columns: its partial is
// written out and merged (the merge participants wait for the block's last piece).
constexpr int64_t PF_SPLIT_COST = 3;
// With clusters: extra cost of a piece of a block split over one cluster's columns (its
// partial staged in shared memory and merged over distributed shared memory).
constexpr int64_t PF_CLUSTER_MERGE_COST = 2;

// The smallest budget T in [t_lo, t_hi] with columns(T) <= gx, given that t_hi is
// feasible: every thread of the CTA tries its own candidate, in two rounds (the
// second within the step of the first); t_lo and t_hi live in shared memory and
// end with t_hi = the answer.  scan: blockDim.x ints of shared memory.
template <class Cols>
__device__ void smallest_budget(Cols columns, int64_t gx, long long &t_lo_s, long long &t_hi_s, int32_t *scan) {
    const int32_t tid = threadIdx.x;
    for (int32_t round = 0; round < 2; ++round) {
        const int64_t t_lo = t_lo_s, t_hi = t_hi_s;
        const int64_t step = max((int64_t)1, (t_hi - t_lo + blockDim.x) / (int64_t)blockDim.x);
        const int64_t T = t_lo + (int64_t)tid * step;
        const bool feas = T <= t_hi && columns(T) <= gx;
        // the smallest feasible candidate (candidates increase with tid)
        scan[tid] = feas ? tid : (int32_t)blockDim.x;
        __syncthreads();
        for (int32_t d = (int32_t)blockDim.x / 2; d > 0; d >>= 1) {
            if (tid < d) scan[tid] = min(scan[tid], scan[tid + d]);
            __syncthreads();
        }
        if (tid == 0) {
            const int32_t w = scan[0];
            if (w < (int32_t)blockDim.x) {
                t_hi_s = t_lo + (int64_t)w * step;   // feasible
                t_lo_s = w > 0 ? t_lo + (int64_t)(w - 1) * step + 1 : t_lo;
            } else {
                t_lo_s = t_lo + (int64_t)(blockDim.x - 1) * step + 1;
            }
        }
        __syncthreads();
    }
}

// cta0[x] = the first item of column >= x, cta0[gx] = n_items (items in column
// order; every thread of the CTA takes part).
__device__ void fill_cta0(const kvk::WorkItem *work, int32_t n_items, int64_t gx, int32_t *cta0) {
    for (int32_t i = threadIdx.x; i < n_items; i += blockDim.x) {
        const int32_t c = work[i].cta;
        const int32_t cp = i > 0 ? work[i - 1].cta : -1;
        for (int32_t x = cp + 1; x <= c; ++x) cta0[x] = i;
    }
    const int32_t clast = n_items > 0 ? work[n_items - 1].cta : -1;
    for (int32_t x = clast + 1 + (int32_t)threadIdx.x; x <= (int32_t)gx; x += blockDim.x) cta0[x] = n_items;
}

__global__ void __launch_bounds__(1024) k_plan_work(kvk::UbView u, kvk::Plan p, int32_t gx_dec, int32_t gx_pf) {
    __shared__ long long t_lo_s, t_hi_s;
    __shared__ int32_t scan_i[1024];
    __shared__ int32_t s_wc[DEC_STAGE];
    __shared__ int32_t s_r0[kvk::PLAN_MAX_COLS], s_nq[kvk::PLAN_MAX_COLS];
    __shared__ long long s_load[kvk::PLAN_MAX_COLS];
    const int32_t tid = threadIdx.x;
    for (int32_t pass = 0; pass < 2; ++pass) {
        const int32_t lo = pass == 0 ? 0 : u.n_dec_blocks;
        const int32_t hi = pass == 0 ? u.n_dec_blocks : u.n_blocks;
        const int64_t gx = pass == 0 ? gx_dec : gx_pf;
        const int32_t item_base = pass == 0 ? 0 : p.cap_dec;
        const int32_t cap = pass == 0 ? p.cap_dec : p.cap_pf;
        int32_t *cta0 = p.cta_item0 + (pass == 0 ? 0 : gx_dec + 1);
        if (lo == hi) {   // no block on this path: its attention kernels are not launched
            if (tid == 0) p.n_work[pass] = 0;
            for (int32_t x = tid; x <= (int32_t)gx; x += blockDim.x) cta0[x] = 0;
            __syncthreads();
            continue;
        }
        if (pass == 1 && p.pf_cluster > 1) {
            // Prefill with clusters of C columns.  A block is either whole (one item)
            // or split into C pieces of equal pair counts, one per column of one
            // cluster, each the last item of its column (its partial stays in shared
            // memory until the cluster merges it).  At most one split block per
            // cluster: the blocks that gain from splitting, largest first; then the
            // whole blocks, largest first, each into the least loaded column.
            if (tid == 0) {
                const int64_t C = p.pf_cluster, Ci = PF_ITEM_COST, D = PF_DIAG_COST, MC = PF_CLUSTER_MERGE_COST;
                const int32_t ncl = (int32_t)(gx / C);
                const int32_t nb = hi - lo;
                auto pairs_of = [&](int32_t b) -> int64_t { return (p.counts[b] + 1) / 2; };
                auto whole_cost = [&](int32_t b) -> int64_t { const int64_t pr = pairs_of(b); return Ci + pr + (pr > 0 ? D : 0); };
                auto piece_cost = [&](int32_t b) -> int64_t { return Ci + (pairs_of(b) + C - 1) / C + D + MC; };
                // scan_i[b - lo]: -2 unplaced, -1 split, else the block's column
                for (int32_t k = 0; k < nb && k < 1024; ++k) scan_i[k] = -2;
                for (int32_t x = 0; x < (int32_t)gx; ++x) {
                    s_load[x] = 0;
                    s_nq[x] = -1;                       // (for now) the cluster's split block
                }
                int32_t nsplit = 0;
                while (nsplit < ncl) {
                    int32_t best = -1;
                    int64_t bw = 0;
                    for (int32_t b = lo; b < hi && b - lo < 1024; ++b) {
                        const int64_t w = whole_cost(b);
                        if (scan_i[b - lo] == -2 && w > piece_cost(b) && w > bw) {
                            best = b;
                            bw = w;
                        }
                    }
                    if (best < 0) break;
                    scan_i[best - lo] = -1;
                    s_nq[nsplit] = best;
                    for (int32_t r = 0; r < (int32_t)C; ++r) s_load[nsplit * C + r] += piece_cost(best);
                    ++nsplit;
                }
                while (true) {
                    int32_t best = -1;
                    int64_t bw = -1;
                    for (int32_t b = lo; b < hi && b - lo < 1024; ++b) {
                        const int64_t w = whole_cost(b);
                        if (scan_i[b - lo] == -2 && w > bw) {
                            best = b;
                            bw = w;
                        }
                    }
                    if (best < 0) break;
                    int32_t xm = 0;
                    for (int32_t x = 1; x < ncl * (int32_t)C; ++x)
                        if (s_load[x] < s_load[xm]) xm = x;
                    scan_i[best - lo] = xm;
                    s_load[xm] += bw;
                }
                // items column by column: the column's whole blocks, then its piece
                int32_t nitem = 0;
                for (int32_t x = 0; x < (int32_t)gx; ++x) {
                    for (int32_t b = lo; b < hi && b - lo < 1024; ++b) {
                        if (scan_i[b - lo] != x) continue;
                        kvk::WorkItem w;
                        w.block = b;
                        w.t0 = 0;
                        w.t1 = p.counts[b];
                        w.cta = x;
                        p.blk_item0[b] = item_base + nitem;
                        p.blk_nitems[b] = 1;
                        if (nitem < cap) p.work[item_base + nitem] = w;
                        else kvd::report(p.err, kvd::DERR_BOUNDS);
                        ++nitem;
                    }
                    const int32_t cl = x / (int32_t)C, r = x % (int32_t)C;
                    const int32_t sb = cl < ncl ? s_nq[cl] : -1;
                    if (sb >= 0) {
                        const int32_t cnt = p.counts[sb];
                        const int64_t pr = pairs_of(sb);
                        kvk::WorkItem w;
                        w.block = sb;
                        // cut in cost, the last pair (the diagonal) costing 1 + D: the piece
                        // holding it gets fewer pairs when the count does not divide evenly
                        auto cut = [&](int64_t k) -> int64_t { return k >= C ? pr : min(pr, k * (pr + D) / C); };
                        w.t0 = (int32_t)min((int64_t)cnt, 2 * cut(r));
                        w.t1 = (int32_t)min((int64_t)cnt, 2 * cut(r + 1));
                        w.cta = x;
                        if (r == 0) {
                            p.blk_item0[sb] = item_base + nitem;
                            p.blk_nitems[sb] = (int32_t)C;
                        }
                        if (nitem < cap) p.work[item_base + nitem] = w;
                        else kvd::report(p.err, kvd::DERR_BOUNDS);
                        ++nitem;
                    }
                }
                if (nb > 1024) kvd::report(p.err, kvd::DERR_BOUNDS);
                p.n_work[1] = min(nitem, cap);
            }
            __syncthreads();   // items written by thread 0 are visible below
        } else if (pass == 1) {
            // Prefill: work in pairs of tiles, PF_ITEM_COST per item, plus PF_DIAG_COST
            // for the piece holding a block's last pair.
            const int64_t C = PF_ITEM_COST, D = PF_DIAG_COST, MS = PF_SPLIT_COST;
            // the blocks' tile counts, staged for the budget search
            for (int32_t b = lo + tid; b < hi && b - lo < DEC_STAGE; b += blockDim.x) s_wc[b - lo] = p.counts[b];
            __syncthreads();
            auto count_of = [&](int32_t b) -> int32_t { return b - lo < DEC_STAGE ? s_wc[b - lo] : p.counts[b]; };
            // how much of the rest of a block a column with `room` left takes: all of
            // it when its diagonal fits too (plus the merge cost when the block is
            // already split), else as much as fits short of the last pair, which splits
            // the block (0: nothing fits, start a new column)
            auto take_of = [&](int64_t rem, int64_t room, bool split, int64_t &cost) -> int64_t {
                const int64_t pen = split ? MS : 0;
                if (rem + D + pen <= room) {
                    cost = rem + D + pen;
                    return rem;
                }
                const int64_t t = min(rem - 1, room - MS);
                if (t < 1) return 0;
                cost = t + MS;
                return t;
            };
            if (tid == 0) {
                int64_t P = 0;
                int32_t nne = 0;
                for (int32_t b = lo; b < hi; ++b) {
                    const int64_t pr = (count_of(b) + 1) / 2;
                    P += pr;
                    nne += pr > 0 ? 1 : 0;
                }
                t_lo_s = max(C + D + 1, (P + (C + D) * nne + gx - 1) / gx);   // lower bound on T
                t_hi_s = P + (C + D) * (nne + 1) + 1;                       // feasible with any gx >= 1
            }
            __syncthreads();
            // columns the greedy fill needs with budget T (stops counting past gx)
            auto columns = [&](int64_t T) -> int64_t {
                int64_t x = 0, acc = 0;
                for (int32_t b = lo; b < hi && x < gx; ++b) {
                    const int64_t pairs = (count_of(b) + 1) / 2;
                    int64_t done = 0;
                    bool split = false;
                    while (done < pairs && x < gx) {
                        int64_t cost = 0;
                        const int64_t room = T - acc - C;
                        const int64_t take = room < 1 ? 0 : take_of(pairs - done, room, split, cost);
                        if (take < 1) {
                            ++x;
                            acc = 0;
                            continue;
                        }
                        if (take < pairs - done) split = true;
                        done += take;
                        acc += C + cost;
                    }
                }
                return x + 1;
            };
            smallest_budget(columns, gx, t_lo_s, t_hi_s, scan_i);
            if (tid == 0) {
                const int64_t T = t_hi_s;
                int32_t x = 0, nitem = 0;
                int64_t acc = 0;
                auto emit = [&](int32_t b, int32_t t0, int32_t t1) {
                    kvk::WorkItem w;
                    w.block = b;
                    w.t0 = t0;
                    w.t1 = t1;
                    w.cta = x;
                    if (nitem < cap) p.work[item_base + nitem] = w;
                    else kvd::report(p.err, kvd::DERR_BOUNDS);
                    ++nitem;
                };
                for (int32_t b = lo; b < hi; ++b) {
                    const int32_t cnt = count_of(b);
                    const int64_t pairs = (cnt + 1) / 2;
                    p.blk_item0[b] = item_base + nitem;
                    int32_t nseg = 0;
                    if (pairs == 0) {
                        emit(b, 0, 0);
                        nseg = 1;
                    } else {
                        int64_t done = 0;
                        bool split = false;
                        while (done < pairs) {
                            int64_t cost = 0;
                            const int64_t room = T - acc - C;
                            int64_t take = room < 1 ? 0 : take_of(pairs - done, room, split, cost);
                            if (take < 1 && x < gx - 1) {   // this column is full
                                ++x;
                                acc = 0;
                                continue;
                            }
                            if (x == gx - 1) {              // the last column takes the rest
                                take = pairs - done;
                                cost = take + D + (split ? MS : 0);
                            }
                            if (take < pairs - done) split = true;
                            emit(b, (int32_t)(2 * done), (int32_t)min((int64_t)cnt, 2 * (done + take)));
                            ++nseg;
                            done += take;
                            acc += C + cost;
                        }
                    }
                    p.blk_nitems[b] = nseg;
                }
                p.n_work[1] = min(nitem, cap);
            }
            __syncthreads();   // items written by thread 0 are visible below
        }
        if (pass == 1) {
            fill_cta0(p.work + item_base, p.n_work[1], gx, cta0);
            __syncthreads();
            // each column's first item: its first pair (TMA rows of its two tiles, fully
            // visible?), and its block's first row and query-vector count, staged for the
            // row table below
            for (int32_t x = tid; x < (int32_t)gx; x += blockDim.x) {
                const int32_t i = cta0[x];
                int32_t f[4] = {-1, -1, 0, 0};
                int32_t r0 = 0, nq = 0;
                if (i < cta0[x + 1]) {
                    const kvk::WorkItem w = p.work[item_base + i];
                    const kvi::DevBlock b = u.blocks[w.block];
                    r0 = b.row0;
                    nq = b.n_rows * p.gqa;
                    if (w.t1 > w.t0) {
                        const int32_t *list = p.tiles + (int64_t)w.block * p.tile_stride;
                        const uint32_t *flg = p.flags + (int64_t)w.block * p.tile_stride;
                        bool full = true;
                        for (int h = 0; h < 2; ++h) {
                            const int32_t t = w.t0 + h < w.t1 ? list[w.t0 + h] : -1;
                            f[h] = t >= 0 ? b.stream * u.kv_size + t * TILE : -TILE;
                            full = full && t >= 0 && (int32_t)(flg[t] & 0xffffu) == b.n_rows * TILE;
                        }
                        f[2] = full ? 1 : 0;
                    }
                }
                for (int h = 0; h < 4; ++h) p.pf_first[4 * x + h] = f[h];
                s_r0[x] = r0;
                s_nq[x] = nq;
            }
            __syncthreads();
            // the rows behind each column's first item, one entry per query vector
            for (int32_t e = tid; e < (int32_t)gx * kvi::PF_M; e += blockDim.x) {
                const int32_t x = e / kvi::PF_M, qv = e % kvi::PF_M;
                p.pf_rows[e] = qv < s_nq[x] ? u.perm[s_r0[x] + qv / p.gqa] : -1;
            }
            continue;
        }
        // Decode: work in the tile costs (the cumulative costs of k_plan_compact),
        // DEC_ITEM_COST per item.  Items are cut in cost units and turned into tile
        // ranges afterwards (equal offsets give equal tiles, so neighbouring items
        // still meet exactly).
        const int64_t C = DEC_ITEM_COST, MT = DEC_MIN_TAKE;
        for (int32_t b = lo + tid; b < hi && b - lo < DEC_STAGE; b += blockDim.x) s_wc[b - lo] = p.wcount[b];
        __syncthreads();
        auto wc = [&](int32_t b) -> int64_t { return b - lo < DEC_STAGE ? s_wc[b - lo] : p.wcount[b]; };
        // how much of a block's remaining cost `rem` a column with `room` left takes
        // (0: none, start a new column)
        auto take_of = [&](int64_t rem, int64_t room) -> int64_t { return room >= min(rem, MT) ? min(rem, room) : 0; };
        if (tid == 0) {
            int64_t S = 0;
            for (int32_t b = lo; b < hi; ++b) S += wc(b);
            const int64_t nb = hi - lo;
            t_lo_s = max(C + MT, (S + C * nb + gx - 1) / gx);   // lower bound on T
            t_hi_s = max(C + MT, S + C * (nb + 1) + 1);         // one column takes everything
        }
        __syncthreads();
        // columns the greedy fill needs with budget T (stops counting past gx)
        auto columns = [&](int64_t T) -> int64_t {
            int64_t x = 0, acc = 0;
            for (int32_t b = lo; b < hi && x < gx; ++b) {
                int64_t rem = wc(b);
                if (rem == 0) {   // an empty item
                    if (acc > 0 && acc + C > T) {
                        ++x;
                        acc = 0;
                    }
                    acc += C;
                    continue;
                }
                while (rem > 0 && x < gx) {
                    const int64_t take = take_of(rem, T - acc - C);
                    if (take == 0) {
                        ++x;
                        acc = 0;
                        continue;
                    }
                    rem -= take;
                    acc += C + take;
                }
            }
            return x + 1;
        };
        smallest_budget(columns, gx, t_lo_s, t_hi_s, scan_i);
        if (tid == 0) {
            const int64_t T = t_hi_s;
            int32_t x = 0, nitem = 0;
            int64_t acc = 0;
            auto emit = [&](int32_t b, int64_t c0, int64_t c1) {   // cost offsets, for now
                kvk::WorkItem w;
                w.block = b;
                w.t0 = (int32_t)c0;
                w.t1 = (int32_t)c1;
                w.cta = x;
                if (nitem < cap) p.work[item_base + nitem] = w;
                else kvd::report(p.err, kvd::DERR_BOUNDS);
                ++nitem;
            };
            for (int32_t b = lo; b < hi; ++b) {
                int64_t rem = wc(b), off = 0;
                p.blk_item0[b] = item_base + nitem;
                int32_t nseg = 0;
                if (rem == 0) {
                    if (acc > 0 && acc + C > T && x < gx - 1) {
                        ++x;
                        acc = 0;
                    }
                    emit(b, 0, 0);
                    acc += C;
                    nseg = 1;
                }
                while (rem > 0) {
                    int64_t take = take_of(rem, T - acc - C);
                    if (take == 0 && x < gx - 1) {   // this column is full
                        ++x;
                        acc = 0;
                        continue;
                    }
                    if (x == gx - 1) take = rem;     // the last column takes the rest
                    emit(b, off, off + take);
                    ++nseg;
                    off += take;
                    rem -= take;
                    acc += C + take;
                }
                p.blk_nitems[b] = nseg;
            }
            p.n_work[0] = min(nitem, cap);
        }
        __syncthreads();   // items written by thread 0 are visible below
        const int32_t n_items = p.n_work[0];
        for (int32_t i = tid; i < n_items; i += blockDim.x) {
            kvk::WorkItem &w = p.work[item_base + i];
            if (w.t1 > w.t0) {
                const int32_t t0 = tile_at_cost(p, w.block, w.t0), t1 = tile_at_cost(p, w.block, w.t1);
                w.t0 = t0;
                w.t1 = t1;
            }
        }
        __syncthreads();   // items written by other threads are visible below
        fill_cta0(p.work + item_base, n_items, gx, cta0);
        __syncthreads();
        // each column's start record (see Plan::dec_first)
        for (int32_t x = tid; x < (int32_t)gx; x += blockDim.x) {
            int32_t f[kvk::DEC_FIRST];
            for (int h = 0; h < kvk::DEC_FIRST; ++h) f[h] = -1;
            if (cta0[x] < cta0[x + 1]) {
                const kvk::WorkItem w = p.work[item_base + cta0[x]];
                const kvi::DevBlock b = u.blocks[w.block];
                const int32_t *list = p.tiles + (int64_t)w.block * p.tile_stride;
                const uint32_t *flg = p.flags + (int64_t)w.block * p.tile_stride;
                for (int h = 0; h < 4; ++h) {
                    const int32_t e = w.t0 + h;
                    if (e < w.t1) {
                        f[h] = list[e];
                        f[4 + h] = (int32_t)flg[f[h]];
                    }
                }
                f[8] = w.block;
                f[9] = w.t0;
                f[10] = w.t1;
                f[11] = b.stream * u.kv_size;
                f[12] = b.n_rows;
                f[13] = b.seq0;
            }
            for (int h = 0; h < kvk::DEC_FIRST; ++h) p.dec_first[kvk::DEC_FIRST * x + h] = f[h];
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) k_mask(kvk::UbView u, uint16_t *mask) {
    const int32_t i = blockIdx.y;
    const int32_t j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= u.n_kv) return;
    const kvi::DevRow r = u.rows[i];
    const int64_t g = (int64_t)r.stream * u.kv_size + j;
    bool vis = u.cell_epoch[g] <= u.ub_epoch;
    if (vis) {
        const uint64_t w = u.cell_bits[g * u.n_words + (r.seq0 >> 6)];
        vis = (w >> (r.seq0 & 63)) & 1ull;
    }
    if (vis) vis = kvd::pos_visible(u.causal, u.n_swa, r.pos, u.cell_pos[g]);
    mask[(int64_t)i * u.n_kv + j] = vis ? (uint16_t)0x0000 : (uint16_t)0xFC00;
}

}  // namespace

namespace kvk {

cudaError_t launch_plan(const UbView &u, const Plan &p, int32_t n_stream, int32_t gx_dec, int32_t gx_pf,
                        cudaStream_t st) {
    const int32_t n_tiles = (u.n_kv + TILE - 1) / TILE;
    const size_t sh = (size_t)u.n_blocks * 2 * sizeof(uint32_t);
    if (sh > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_plan_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sh);
        if (e != cudaSuccess) return e;
    }
    k_plan_tiles<<<dim3(n_tiles, n_stream), TILE, sh, st>>>(u, p);
    k_plan_compact<<<u.n_blocks, 256, 0, st>>>(u, p, n_tiles);
    k_plan_work<<<1, 1024, 0, st>>>(u, p, gx_dec, gx_pf);
    return cudaGetLastError();
}

cudaError_t load_plan_kernels() {
    cudaFuncAttributes fa;
    cudaError_t e;
    if ((e = cudaFuncGetAttributes(&fa, k_plan_tiles)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, k_plan_compact)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, k_plan_work)) != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, k_mask);
}

cudaError_t launch_mask(const UbView &u, uint16_t *mask, cudaStream_t st) {
    k_mask<<<dim3((u.n_kv + 255) / 256, u.n_tokens), 256, 0, st>>>(u, mask);
    return cudaGetLastError();
}

}  // namespace kvk
