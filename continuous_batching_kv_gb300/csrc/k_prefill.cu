// K3b: GQA flash attention, prefill / mixed path, on tcgen05 tensor cores.
//
// "llama.cpp and the ubatch", "Chunked prefill is the same mechanism": a
// chunk of U rows against C cached cells is a [U, C+U] score matrix; with the
// mask of "The mask is doing the work" (occupied, same first sequence id,
// not later) it is the same softmax(q K^T / sqrt(d) + mask) V as decode, but
// now a dense contraction worth putting on the tensor cores.
//
// Design (sm_103a, one CTA of 320 threads per SM):
//  * a block = up to 128 query vectors (rows sharing a stream and first
//    sequence id, times the GQA group) = the 128 TMEM lanes of one MMA tile;
//    a work item = one block, one KV head, a chunk of the block's list of
//    visible 64-cell tiles, consumed two at a time (N = 128 cells);
//  * warp 8 streams K and V tiles with TMA (128-byte swizzle) into separate
//    2-slot K and V rings, with each pair's list entries, flags and per-cell
//    visibility fetched ahead into a metadata ring; warp 9 allocates TMEM and
//    one thread issues
//    tcgen05.mma: S = Q K^T (M 128, N 128, K 128) into one of two TMEM score
//    buffers as soon as the softmax has read that buffer, and O += P V with P
//    read from TMEM (double-buffered, fp16) and V MN-major from shared memory
//    into a TMEM accumulator; tcgen05.commit signals the mbarriers;
//  * warps 0-7 (two threads per TMEM lane = query vector, 64 columns each)
//    read S with one tcgen05.ld as soon as it lands (TMEM reads stall behind
//    running MMAs), apply the mask per cell on tiles that are not fully
//    visible, run the online softmax in base 2 (a quarter of the exponentials
//    on the FMA pipe), write P (fp16, two cells per 32-bit column) into the
//    TMEM P buffer of the pair's parity, and rescale O in TMEM only when the
//    running maximum grew by more
//    than 2^8 (otherwise the stale maximum is kept; the final normalisation
//    uses the same one);
//  * cells nobody in the block may see get their V rows zeroed in shared
//    memory before the PV product (P is 0 there, but 0 * NaN would not be);
//  * a block split over several CTAs leaves one partial (m, l, O) per piece,
//    merged by a small second kernel, so no CTA stalls its own pipeline to
//    merge; every mbarrier wait is bounded.

#include "dev_common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace {

using kvi::TILE;

constexpr int NSM = 256;                 // softmax threads: two per TMEM lane
constexpr int NT = NSM + 64;             // + producer warp + MMA warp
constexpr int M = 128;
constexpr int HALF = 128 * 128;          // [128 rows][64 fp16], 128-byte rows
constexpr int TILEB = 2 * HALF;          // 32 KiB
constexpr int BOX = 64 * 128;            // one TMA box: 64 rows x 64 fp16
constexpr int STAGES = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILEB;
constexpr int OFF_V = OFF_K + STAGES * TILEB;
constexpr int OFF_AUX = OFF_V + STAGES * TILEB;
constexpr int PART_STRIDE = 132;
constexpr uint32_t TMEM_COLS = 512;      // S0 [0,128), S1 [128,256), O [256,384), P0, P1 [384,512)
constexpr uint32_t COL_O = 256;
constexpr uint32_t COL_P = 384;          // P of pair g: fp16, 64 columns at COL_P + 64 (g & 1)
constexpr float RESCALE_LOG2 = 8.0f;
constexpr unsigned POLL_NS = 32;         // back-off of the polling producer / MMA loops

constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16(128, 128, 0, 1);

// Metadata ring.  Pair g's slot is rewritten by the K load of pair g + 8, which
// needs S of g + 6, which needs the softmax to have read S of g + 4: by then the
// softmax is done with pair g, and PV of g (hence the V load of g, which reads
// the slot) was issued before the softmax of g + 2 wrote its P.
constexpr int MSLOTS = 8;

struct Meta {                 // per pair tile: what the producer learned about it
    int32_t full;
    int32_t ys[2];            // TMA row coordinates of the two 64-cell halves
    int32_t pad;
    int32_t cpos[128];
    uint8_t has[128];         // cell holds the block's sequence and is not from a later ubatch
    uint8_t anyvis[128];      // ... and some row of the block may see it
};

struct ItemSlot {             // per work item: the query vector behind each TMEM lane
    int32_t row[M];           // ubatch row, -1 for lanes past the block's query vectors
    int32_t rpos[M];
};

struct __align__(16) Aux {
    uint64_t k_full[STAGES], v_full[STAGES], k_empty[STAGES], v_empty[STAGES];
    uint64_t meta_full[MSLOTS];
    uint64_t s_full[2], p_full[2], pv_done[2], q_full, spare;   // p_full, pv_done [g & 1]: pair g
    uint64_t s_free[2];       // a score buffer was read into registers by all 256 softmax threads
    uint64_t rbar, lbar;      // softmax-group exchanges (row maxima, row sums), all 256 threads
    uint32_t tmem_base;
    int32_t fail;
    int32_t flag;
    int32_t pad;
    Meta meta[MSLOTS];
    ItemSlot islot[2];
    float red[2][2][M];       // [pair parity][column half][row]: partial row maxima
    float lex[2][2][M];       // [item parity][column half][row]: partial row sums
};

constexpr size_t SMEM_BYTES = OFF_AUX + sizeof(Aux);

__device__ __forceinline__ bool wait_or_fail(uint64_t *bar, uint32_t parity, volatile int32_t *fail) {
    if (kvd::mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (!kvd::mbar_try_wait(bar, parity)) {
        if (*fail) return false;
        if (clock64() - t0 > kvd::WAIT_LIMIT_CYCLES) {
            *fail = 1;
            return false;
        }
    }
    return true;
}

// 2^x with the hardware's approximate base-2 exponential (ex2.approx.ftz:
// flushes subnormals, 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^x on the FMA pipe.  Range reduction: x = n + f with n = round(x) taken by
// adding 1.5 * 2^23 (the integer lands in the low mantissa bits), f in
// [-1/2, 1/2]; 2^f by a cubic 1 + f (c1 + f (c2 + f c3)) whose coefficients
// were fitted here to minimise the maximum relative error on [-1/2, 1/2]
// (about 1.0e-4, below the 4.9e-4 half-ulp of the fp16 P it feeds); 2^n is
// added to the exponent field with one integer multiply-add.  x is clamped to
// -127, where the result is exactly +0 (so is 2^-inf).
__device__ __forceinline__ float ex2_poly(float x) {
    constexpr float MAGIC = 12582912.0f;    // 1.5 * 2^23
    constexpr float C1 = 6.932828051e-01f, C2 = 2.422090319e-01f, C3 = 5.500809860e-02f;
    x = fmaxf(x, -127.0f);
    const float t = x + MAGIC;
    const float nf = t - MAGIC;
    const float f = x - nf;
    const float p = fmaf(f, fmaf(f, fmaf(f, C3, C2), C1), 1.0f);
    return __uint_as_float(__float_as_uint(p) + (__float_as_uint(t) << 23));
}

// True while no wait has given up, agreed by all 32 lanes of the warp (so a
// failure never splits a warp in front of a warp-collective instruction).
__device__ __forceinline__ bool warp_ok(volatile int32_t *fail) { return __all_sync(0xffffffffu, *fail == 0); }

struct ItemInfo {
    int32_t block, t0, t1, pairs, nitems;
};

__device__ __forceinline__ ItemInfo item_info(const kvk::PrefillArgs &a, int32_t wi) {
    const kvk::WorkItem w = a.p.work[a.p.cap_dec + wi];
    ItemInfo r;
    r.block = w.block;
    r.t0 = w.t0;
    r.t1 = w.t1;
    r.pairs = (w.t1 - w.t0 + 1) / 2;
    r.nitems = a.p.blk_nitems[w.block];
    return r;
}

__global__ void __launch_bounds__(NT, 1)
k_prefill(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
          const kvk::PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Aux &x = *reinterpret_cast<Aux *>(smem + OFF_AUX);
    volatile int32_t *fail = &x.fail;
    const int32_t tid = threadIdx.x;
    const int32_t warp = tid >> 5;
    const int32_t hk = blockIdx.y;
    const int32_t G = a.gqa;
    const int32_t* c0 = a.p.cta_item0 + a.gx_dec + 1;
    const int32_t i0 = c0[blockIdx.x];
    const int32_t i1 = c0[blockIdx.x + 1];
    const uint32_t sbase = kvd::smem_u32(smem);

    if ((sbase & 1023u) != 0) {
        if (tid == 0) kvd::report(a.err, kvd::DERR_BOUNDS);
        return;
    }
    if (tid == 0) {
        kvd::prefetch_tmap(&tm_k);
        kvd::prefetch_tmap(&tm_v);
        for (int s = 0; s < STAGES; ++s) {
            kvd::mbar_init(&x.k_full[s], 1);
            kvd::mbar_init(&x.v_full[s], 1);
            kvd::mbar_init(&x.k_empty[s], 1);
            kvd::mbar_init(&x.v_empty[s], 1);
        }
        for (int s = 0; s < MSLOTS; ++s) kvd::mbar_init(&x.meta_full[s], 32);
        kvd::mbar_init(&x.s_full[0], 1);
        kvd::mbar_init(&x.s_full[1], 1);
        kvd::mbar_init(&x.s_free[0], NSM);
        kvd::mbar_init(&x.s_free[1], NSM);
        kvd::mbar_init(&x.p_full[0], NSM);
        kvd::mbar_init(&x.p_full[1], NSM);
        kvd::mbar_init(&x.pv_done[0], 1);
        kvd::mbar_init(&x.pv_done[1], 1);
        kvd::mbar_init(&x.q_full, NSM);
        kvd::mbar_init(&x.spare, 1);
        kvd::mbar_init(&x.rbar, NSM);
        kvd::mbar_init(&x.lbar, NSM);
        x.fail = 0;
        kvd::fence_mbar_init();
    }
    if (warp == 9) {
        tc::alloc(&x.tmem_base, TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = x.tmem_base;

    if (warp == 8) {
        // ===================== producer (whole warp) =====================
        // K and V tiles live in separate 2-slot rings: K of pair g + 2 loads as soon
        // as S of pair g has consumed K of g; V of g + 2 as soon as PV of g is done.
        // Two cursors walk the CTA's pair sequence; whichever load may go is issued
        // (decisions by lane 0, broadcast), nothing waits on one while the other is
        // ready.  The K load also publishes the pair's metadata (and, for an item's
        // first pair, its lane table) through meta_full.
        const int32_t lane = tid & 31;
        int32_t total = 0;
        for (int32_t wi = i0; wi < i1; ++wi) total += item_info(a, wi).pairs;
        int32_t kc = 0, vc = 0, nonempty = 0;
        int32_t kwi = i0, kj = 0;              // K cursor: item and pair within it
        ItemInfo kit{};
        kvi::DevBlock kb{};
        bool have_k = false;
        int32_t tt[2] = {-1, -1};
        bool full = false;
        bool mhas[4] = {false, false, false, false}, many[4] = {false, false, false, false};
        int32_t mpos[4] = {0, 0, 0, 0}, lrow[4] = {-1, -1, -1, -1}, lpos[4] = {0, 0, 0, 0};
        long long t_last = clock64();
        while (vc < total) {
            if (!warp_ok(fail)) break;
            bool prog = false;
            if (kc < total) {
                if (!have_k) {
                    // the next K load's global reads, done before its slot is free
                    while (true) {
                        kit = item_info(a, kwi);
                        if (kj < kit.pairs) break;
                        ++kwi;
                        kj = 0;
                    }
                    kb = a.u.blocks[kit.block];
                    const int32_t *list = a.p.tiles + (int64_t)kit.block * a.p.tile_stride;
                    const uint32_t *flg = a.p.flags + (int64_t)kit.block * a.p.tile_stride;
                    bool fullh[2];
                    for (int h = 0; h < 2; ++h) {
                        const int32_t e = kit.t0 + 2 * kj + h;
                        tt[h] = e < kit.t1 ? list[e] : -1;
                        fullh[h] = tt[h] >= 0 && (int32_t)(flg[tt[h]] & 0xffffu) == kb.n_rows * TILE;
                    }
                    full = fullh[0] && fullh[1];
                    if (!full) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int32_t c = lane + 32 * r;
                            const int32_t t = tt[c >> 6];
                            bool has = false;
                            int32_t cp = 0;
                            if (t >= 0) {
                                const int32_t jc = t * TILE + (c & 63);
                                if (jc < a.u.n_kv) {
                                    const int64_t g = (int64_t)kb.stream * a.u.kv_size + jc;
                                    const uint64_t w = a.u.cell_bits[g * a.u.n_words + (kb.seq0 >> 6)];
                                    has = ((w >> (kb.seq0 & 63)) & 1ull) && a.u.cell_epoch[g] <= a.u.ub_epoch;
                                    cp = a.u.cell_pos[g];
                                }
                            }
                            mhas[r] = has;
                            mpos[r] = cp;
                            many[r] = has && (!a.u.causal || cp <= kb.pos_max);
                        }
                    }
                    if (kj == 0) {
                        const int32_t nqv = kb.n_rows * G;
                        for (int r = 0; r < 4; ++r) {
                            const int32_t n = lane + 32 * r;
                            lrow[r] = -1;
                            lpos[r] = 0;
                            if (n < nqv) {
                                lrow[r] = a.u.perm[kb.row0 + n / G];
                                lpos[r] = a.u.rows[lrow[r]].pos;
                            }
                        }
                    }
                    have_k = true;
                }
                const int32_t st = kc % STAGES;
                bool ready = kc < STAGES ||
                             kvd::mbar_test_wait(&x.k_empty[st], (uint32_t)((kc / STAGES) - 1) & 1u);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    Meta &mt = x.meta[kc % MSLOTS];
                    if (kj == 0) {
                        // the item's lane table; its previous reader (two non-empty items
                        // back) read it before any of its S products, and this K slot
                        // was just freed by such an S product
                        ItemSlot &is = x.islot[nonempty & 1];
                        for (int r = 0; r < 4; ++r) {
                            is.row[lane + 32 * r] = lrow[r];
                            is.rpos[lane + 32 * r] = lpos[r];
                        }
                        ++nonempty;
                    }
                    if (lane == 0) {
                        for (int h = 0; h < 2; ++h)   // a missing second tile: out of bounds, TMA writes zeros
                            mt.ys[h] = tt[h] >= 0 ? kb.stream * a.u.kv_size + tt[h] * TILE : -TILE;
                        mt.full = full ? 1 : 0;
                        uint8_t *ks = smem + OFF_K + st * TILEB;
                        const int32_t xk = hk * 128;
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive_expect_tx(&x.k_full[st], TILEB);
                        for (int h = 0; h < 2; ++h) {
                            kvd::tma_load_2d(ks + h * BOX, &tm_k, xk, mt.ys[h], &x.k_full[st]);
                            kvd::tma_load_2d(ks + HALF + h * BOX, &tm_k, xk + 64, mt.ys[h], &x.k_full[st]);
                        }
                    }
                    if (!full) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int32_t c = lane + 32 * r;
                            mt.has[c] = mhas[r] ? 1 : 0;
                            mt.cpos[c] = mpos[r];
                            mt.anyvis[c] = many[r] ? 1 : 0;
                        }
                    }
                    __syncwarp();
                    kvd::mbar_arrive(&x.meta_full[kc % MSLOTS]);
                    ++kc;
                    ++kj;
                    have_k = false;
                    prog = true;
                }
            }
            if (vc < kc) {
                const int32_t st = vc % STAGES;
                bool ready = vc < STAGES ||
                             kvd::mbar_test_wait(&x.v_empty[st], (uint32_t)((vc / STAGES) - 1) & 1u);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    if (lane == 0) {
                        const Meta &mt = x.meta[vc % MSLOTS];   // still intact (see MSLOTS)
                        uint8_t *vs = smem + OFF_V + st * TILEB;
                        const int32_t xk = hk * 128;
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive_expect_tx(&x.v_full[st], TILEB);
                        for (int h = 0; h < 2; ++h) {
                            kvd::tma_load_2d(vs + h * BOX, &tm_v, xk, mt.ys[h], &x.v_full[st]);
                            kvd::tma_load_2d(vs + HALF + h * BOX, &tm_v, xk + 64, mt.ys[h], &x.v_full[st]);
                        }
                    }
                    __syncwarp();
                    ++vc;
                    prog = true;
                }
            }
            if (prog) {
                t_last = clock64();
            } else if (__shfl_sync(0xffffffffu, clock64() - t_last > kvd::WAIT_LIMIT_CYCLES ? 1 : 0, 0)) {
                if (lane == 0) *fail = 1;
                break;
            } else {
                __nanosleep(POLL_NS);   // leave the issue slots to the softmax warps
            }
        }
        if (*fail && lane == 0) {
            // let loads already issued land before the CTA exits
            for (int32_t q = kc > STAGES ? kc - STAGES : 0; q < kc; ++q)
                (void)kvd::mbar_wait_bounded(&x.k_full[q % STAGES], (uint32_t)(q / STAGES) & 1u);
            for (int32_t q = vc > STAGES ? vc - STAGES : 0; q < vc; ++q)
                (void)kvd::mbar_wait_bounded(&x.v_full[q % STAGES], (uint32_t)(q / STAGES) & 1u);
        }
    } else if (warp == 9) {
        // ===================== MMA issuer =====================
        if ((tid & 31) == 0) {
            int32_t gidx = 0;          // global pair-tile counter (stage ring)
            uint32_t s_uses[2] = {0, 0};   // S products written into each score buffer so far
            uint32_t n_q = 0;
            uint32_t n_s[2] = {0, 0};
            const uint32_t q_addr = sbase + OFF_Q;
            auto issue_s = [&](int32_t gi, int32_t buf) {
                const uint32_t k_addr = sbase + OFF_K + (gi % STAGES) * TILEB;
                const uint32_t d = tmem + (uint32_t)buf * 128u;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF + (uint32_t)(kk & 3) * 32u;
                    tc::mma_ss(d, tc::sdesc_sw128(q_addr + off, 16, 1024), tc::sdesc_sw128(k_addr + off, 16, 1024),
                               IDESC_S, kk > 0 ? 1u : 0u);
                }
                tc::commit(&x.s_full[buf]);
                tc::commit(&x.k_empty[gi % STAGES]);   // this K tile is consumed
            };
            // Per item, a non-blocking scheduler: PV of the oldest ready P first (the
            // softmax waits on it), then S of the next pair once its K tile has
            // landed and its score buffer is free (the P two pairs back was taken).
            // Nothing blocks on one condition while the other is ready.
            for (int32_t wi = i0; wi < i1 && !*fail; ++wi) {
                const ItemInfo it = item_info(a, wi);
                if (it.pairs == 0) continue;
                if (!wait_or_fail(&x.q_full, n_q & 1u, fail)) break;
                ++n_q;
                tc::fence_after();
                bool ok = true;
                int32_t s_done = 0, pv_done = 0;
                long long t_last = clock64();
                while (pv_done < it.pairs) {
                    bool progressed = false;
                    // P of pair gi in buffer gi & 1 (a single barrier could be lapped: the
                    // softmax may finish two pairs before this thread looks)
                    const int32_t gp = gidx + pv_done;
                    if (pv_done < s_done && kvd::mbar_test_wait(&x.p_full[gp & 1], (uint32_t)(gp >> 1) & 1u)) {
                        const int32_t gi = gp;
                        ok = wait_or_fail(&x.v_full[gi % STAGES], (uint32_t)(gi / STAGES) & 1u, fail);
                        if (!ok) break;
                        tc::fence_after();
                        const uint32_t v_addr = sbase + OFF_V + (gi % STAGES) * TILEB;
                        const uint32_t p_tmem = tmem + COL_P + 64u * (uint32_t)(gi & 1);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {   // K = 16 cells = 8 TMEM columns of P
                            const uint32_t boff = (uint32_t)kk * 2048u;
                            tc::mma_ts(tmem + COL_O, p_tmem + 8u * (uint32_t)kk,
                                       tc::sdesc_sw128(v_addr + boff, HALF, 1024), IDESC_PV,
                                       (pv_done > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc::commit(&x.pv_done[gi & 1]);
                        tc::commit(&x.v_empty[gi % STAGES]);
                        ++pv_done;
                        progressed = true;
                    }
                    if (s_done < it.pairs) {
                        // S of the next pair: its K tile has landed and its score buffer's
                        // previous contents were read by the softmax
                        const int32_t gi = gidx + s_done;
                        const int32_t buf = s_done & 1;
                        if (kvd::mbar_test_wait(&x.k_full[gi % STAGES], (uint32_t)(gi / STAGES) & 1u) &&
                            (s_uses[buf] == 0 || kvd::mbar_test_wait(&x.s_free[buf], (s_uses[buf] - 1) & 1u))) {
                            tc::fence_after();
                            issue_s(gi, buf);
                            ++n_s[buf];
                            ++s_uses[buf];
                            ++s_done;
                            progressed = true;
                        }
                    }
                    if (progressed) {
                        t_last = clock64();
                    } else if (*fail || clock64() - t_last > kvd::WAIT_LIMIT_CYCLES) {
                        *fail = 1;
                        ok = false;
                        break;
                    } else {
                        __nanosleep(POLL_NS);   // leave the issue slots to the softmax warps
                    }
                }
                gidx += it.pairs;
                if (!ok) break;
            }
            // all issued MMAs complete before TMEM is released
            tc::commit(&x.spare);
            (void)kvd::mbar_wait_bounded(&x.spare, 0);
        }
    } else {
        // ============ softmax / correction / epilogue (warps 0-7, two threads per row) ============
        // Warps w and w + 4 share TMEM lane quarter w: thread (n, ch) owns row n's
        // columns 64ch .. 64ch + 63 of S, P and O.  Row maxima and row sums are
        // combined through shared memory.
        const int32_t n = tid & 127;           // TMEM lane = query vector
        const int32_t ch = tid >> 7;           // column half
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(64 * ch);
        uint32_t n_s[2] = {0, 0};
        uint32_t n_r = 0, n_l = 0;
        int32_t k = 0;                         // pair tiles consumed (stage ring position)
        int32_t nonempty = 0;
        bool ok = true;
        // The two halves of a row meet through mbarriers (arrive, then a bounded
        // wait), never bar.sync: if a wait elsewhere gives up, the others time out
        // instead of waiting for threads that left.
        for (int32_t wi = i0; wi < i1 && ok && warp_ok(fail); ++wi) {
            const ItemInfo it = item_info(a, wi);
            int32_t row = -1, rpos = 0;
            if (it.pairs == 0) {
                // an empty item (its block sees no cell): zeros, or an empty partial
                const kvi::DevBlock b = a.u.blocks[it.block];
                if (n < b.n_rows * G) row = a.u.perm[b.row0 + n / G];
            } else {
                // the first pair's metadata also publishes this item's lane table
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.meta_full[k % MSLOTS], (uint32_t)(k / MSLOTS) & 1u, fail));
                if (!ok) break;
                const ItemSlot &is = x.islot[nonempty & 1];
                ++nonempty;
                row = is.row[n];
                rpos = is.rpos[n];
            }
            const bool live = row >= 0;
            const int32_t h = hk * G + (n % G);
            float *orow = a.o + ((int64_t)(live ? row : 0) * a.n_head + h) * 128 + 64 * ch;
            float m_run = -INFINITY, l_run = 0.f;   // l_run: this thread's half of the row sum
            float ov[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) ov[c] = 0.f;
            if (it.pairs > 0) {
            // ---- Q tile: row n, d-half ch, 128-byte swizzle ----
            {
                uint8_t *qs = smem + OFF_Q + ch * HALF;
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(a.q + ((int64_t)(live ? row : 0) * a.n_head + h) * 128 + 64 * ch);
                uint4 qv[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) qv[c] = live ? src[c] : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(qs + kvd::swz128(n, c)) = qv[c];
                kvd::fence_proxy_async_smem();
                kvd::mbar_arrive(&x.q_full);
            }
            for (int32_t j = 0; j < it.pairs; ++j, ++k) {
                const int32_t st = k % STAGES;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.meta_full[k % MSLOTS], (uint32_t)(k / MSLOTS) & 1u, fail));
                if (!ok) break;
                const Meta &mt = x.meta[k % MSLOTS];
                const bool full = mt.full != 0;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.s_full[j & 1], n_s[j & 1] & 1u, fail));
                if (!ok) break;
                ++n_s[j & 1];
                tc::fence_after();
                // ---- my 64 columns of S -> registers, read from TMEM once, right when
                //      ready (TMEM reads stall behind running MMAs); masked -> -inf ----
                uint32_t sb[64];
                tc::ld64(lane_base + (uint32_t)(j & 1) * 128u, sb);   // warp collective
                tc::fence_before();
                kvd::mbar_arrive(&x.s_free[j & 1]);                   // the next S may overwrite it
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (!live) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) sb[c] = __float_as_uint(-INFINITY);
                } else if (!full) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int cc = 64 * ch + c;
                        const bool vis = mt.has[cc] && (!a.u.causal || mt.cpos[cc] <= rpos);
                        if (!vis) sb[c] = __float_as_uint(-INFINITY);
                    }
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(sb[c]));
                // ---- row maximum over both halves (double-buffered by pair parity) ----
                x.red[j & 1][ch][n] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                kvd::mbar_arrive(&x.rbar);
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.rbar, n_r & 1u, fail));
                ++n_r;
                if (!ok) break;
                const float tmax = fmaxf(x.red[j & 1][0][n], x.red[j & 1][1][n]) * a.scale_log2;
                const float m_new = fmaxf(m_run, tmax);
                const bool grow = m_new > m_run + RESCALE_LOG2 || (m_run == -INFINITY && m_new != -INFINITY);
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2_approx(m_run - m_new);
                    m_run = m_new;
                    l_run *= alpha;
                }
                // ---- P buffer k & 1 is free once PV of pair k - 2 finished (it read it);
                //      that wait is nearly always already satisfied ----
                if (k >= 2) {
                    ok = __all_sync(0xffffffffu,
                                    wait_or_fail(&x.pv_done[k & 1], (uint32_t)((k - 2) >> 1) & 1u, fail));
                    if (!ok) break;
                    tc::fence_after();
                }
                // ---- P = 2^(s*scale - m) as fp16 into TMEM P buffer k & 1: my 64 cells
                //      are 32 columns (two fp16 per column, lower cell in the low half);
                //      one exponential in four on the FMA pipe ----
                {
                    const bool any = m_run != -INFINITY;   // false for lanes past the block
                    const float nm = -m_run;
                    const float sc = a.scale_log2;
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
                    uint32_t pw[32];
#pragma unroll
                    for (int c2 = 0; c2 < 32; ++c2) {
                        const int c = 2 * c2;
                        const float x0 = fmaf(__uint_as_float(sb[c]), sc, nm);
                        const float x1 = fmaf(__uint_as_float(sb[c + 1]), sc, nm);
                        float p0 = ex2_approx(x0);
                        float p1 = (c2 & 1) ? ex2_poly(x1) : ex2_approx(x1);
                        p0 = any ? p0 : 0.f;
                        p1 = any ? p1 : 0.f;
                        ls[c2 & 3] += p0 + p1;
                        __half2 hv = __floats2half2_rn(p0, p1);
                        pw[c2] = *reinterpret_cast<uint32_t *>(&hv);
                    }
                    l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    tc::st32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + COL_P + 64u * (uint32_t)(k & 1) +
                                 32u * (uint32_t)ch, pw);
                }
                // ---- O *= alpha where the running maximum moved (rare), my 64 columns;
                //      O is stable once PV of pair k - 1 finished ----
                if (j > 0 && __any_sync(0xffffffffu, grow)) {
                    ok = __all_sync(0xffffffffu,
                                    wait_or_fail(&x.pv_done[(k - 1) & 1], (uint32_t)((k - 1) >> 1) & 1u, fail));
                    if (!ok) break;
                    tc::fence_after();
#pragma unroll 1
                    for (int q2 = 0; q2 < 2; ++q2) {
                        uint32_t r[32];
                        const uint32_t ta = lane_base + COL_O + (uint32_t)q2 * 32u;
                        tc::ld32(ta, r);
#pragma unroll
                        for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                        tc::st32(ta, r);
                    }
                    tc::wait_st();
                }
                if (!full) {
                    // V rows of cells nobody in the block sees: zero (P is 0 there; V may
                    // be garbage); thread (n, ch) clears d-half ch of cell n
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.v_full[st], (uint32_t)(k / STAGES) & 1u, fail));
                    if (!ok) break;
                    if (!mt.anyvis[n]) {
                        uint8_t *vs = smem + OFF_V + st * TILEB + ch * HALF + n * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(vs + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                tc::wait_st();                     // P (and a rescaled O) are in TMEM
                kvd::fence_proxy_async_smem();     // zeroed V rows are visible to the MMA
                tc::fence_before();
                kvd::mbar_arrive(&x.p_full[k & 1]);
            }
            if (!ok) break;
            // ---- epilogue: wait for the last PV (pair k - 1), read my 64 columns of O ----
            ok = __all_sync(0xffffffffu,
                            wait_or_fail(&x.pv_done[(k - 1) & 1], (uint32_t)((k - 1) >> 1) & 1u, fail));
            if (!ok) break;
            tc::fence_after();
            {
                uint32_t r[64];
                tc::ld64(lane_base + COL_O, r);
#pragma unroll
                for (int c = 0; c < 64; ++c) ov[c] = __uint_as_float(r[c]);
            }
            tc::fence_before();
            }   // it.pairs > 0
            // ---- the row sum over both halves (double-buffered by item parity) ----
            x.lex[n_l & 1][ch][n] = l_run;
            kvd::mbar_arrive(&x.lbar);
            ok = __all_sync(0xffffffffu, wait_or_fail(&x.lbar, n_l & 1u, fail));
            if (!ok) break;
            const float l_tot = x.lex[n_l & 1][0][n] + x.lex[n_l & 1][1][n];
            ++n_l;
            if (it.nitems == 1) {
                if (live) {
                    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll
                    for (int c = 0; c < 64; c += 4)
                        *reinterpret_cast<float4 *>(orow + c) =
                            make_float4(ov[c] * inv, ov[c + 1] * inv, ov[c + 2] * inv, ov[c + 3] * inv);
                }
            } else {
                // a split block: this item's partial (its slot is its index among the
                // prefill items); k_merge_pf combines the partials after the kernel
                float *pp = a.part + (((int64_t)wi * a.n_head_kv + hk) * M + n) * PART_STRIDE;
                if (ch == 0) {
                    pp[0] = m_run;
                    pp[1] = l_tot;
                }
#pragma unroll
                for (int c = 0; c < 64; c += 4)
                    *reinterpret_cast<float4 *>(pp + 4 + 64 * ch + c) = make_float4(ov[c], ov[c + 1], ov[c + 2], ov[c + 3]);
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (*fail && tid == 0) kvd::report(a.err, kvd::DERR_MMA_TIMEOUT);
    if (warp == 9) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
}


// Split-K merge of the prefill path: one CTA per (prefill block, KV head);
// blocks covered by a single item were written directly and return at once.
// Thread t takes row t / 2 and half of its 128 values, so every load is
// independent of the others:  O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q.
__global__ void __launch_bounds__(256) k_merge_pf(const kvk::PrefillArgs a) {
    const int32_t b = a.u.n_dec_blocks + blockIdx.x;
    const int32_t hk = blockIdx.y;
    const int32_t nitems = a.p.blk_nitems[b];
    if (nitems <= 1) return;
    const kvi::DevBlock blk = a.u.blocks[b];
    const int32_t n = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int32_t G = a.gqa;
    if (n >= blk.n_rows * G) return;
    const int32_t row = a.u.perm[blk.row0 + n / G];
    const int32_t h = hk * G + (n % G);
    const int32_t first = a.p.blk_item0[b] - a.p.cap_dec;
    const int64_t istride = (int64_t)a.n_head_kv * M * PART_STRIDE;
    const float *pr = a.part + (((int64_t)first * a.n_head_kv + hk) * M + n) * PART_STRIDE;
    float Mx = -INFINITY;
    for (int32_t q = 0; q < nitems; ++q) Mx = fmaxf(Mx, __ldcg(pr + q * istride));
    float acc[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) acc[c] = 0.f;
    float L = 0.f;
    if (Mx != -INFINITY) {
        for (int32_t q = 0; q < nitems; ++q) {
            const float *pq = pr + q * istride;
            const float mk = __ldcg(pq);
            const float lk = __ldcg(pq + 1);
            float4 v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = __ldcg(reinterpret_cast<const float4 *>(pq + 4 + 64 * half) + c);
            const float sc = mk == -INFINITY ? 0.f : ex2_approx(mk - Mx);
            L = fmaf(lk, sc, L);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                acc[4 * c + 0] = fmaf(v[c].x, sc, acc[4 * c + 0]);
                acc[4 * c + 1] = fmaf(v[c].y, sc, acc[4 * c + 1]);
                acc[4 * c + 2] = fmaf(v[c].z, sc, acc[4 * c + 2]);
                acc[4 * c + 3] = fmaf(v[c].w, sc, acc[4 * c + 3]);
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float *dst = a.o + ((int64_t)row * a.n_head + h) * 128 + 64 * half;
#pragma unroll
    for (int c = 0; c < 16; ++c)
        reinterpret_cast<float4 *>(dst)[c] =
            make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv, acc[4 * c + 2] * inv, acc[4 * c + 3] * inv);
}

}  // namespace

namespace kvk {

cudaError_t launch_prefill(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const PrefillArgs &a,
                           int32_t grid_x, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    k_prefill<<<dim3(grid_x, a.n_head_kv), NT, SMEM_BYTES, st>>>(*tm_k, *tm_v, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_merge_pf<<<dim3(a.u.n_blocks - a.u.n_dec_blocks, a.n_head_kv), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kvk
