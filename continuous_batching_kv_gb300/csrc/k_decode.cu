// K3a: GQA flash attention, decode path (memory bound).
//
// "llama.cpp and the ubatch", "The mask is doing the work" and "Chunked
// prefill is the same mechanism": o = softmax(q K^T / sqrt(d) + mask) V over
// the cells a row may see; masked cells contribute nothing.  "Iteration-Level
// Batching", "The budget that actually binds": the n_head / n_head_kv query
// heads of a group share one KV head.
//
// Design (sm_103a), templated on NQ, the query vectors one block may hold
// (1, 2, 4, 8 or 16; the ubatch's largest decode block picks the instance):
//  * grid = (CTA columns, KV heads), two CTAs per SM; the planner fills the CTA
//    columns with consecutive pieces (work items) of the decode blocks' visible-
//    tile lists, greedily by cost (tiles plus a fixed cost per item) up to the
//    smallest budget that fits the grid, so a column takes a second block only
//    where blocks are small next to the budget; a block is up to
//    16 query vectors (rows sharing a first sequence id, times the GQA group),
//    so every K/V byte read serves all of them;
//  * warp 8 is the producer: K and V of one 64-cell tile per stage, by TMA
//    (2-D tensor maps, 128-byte swizzle), into a 2- or 3-stage ring, with the
//    visibility of the cells of tiles that are not fully visible; its first
//    copy waits for the previous kernel of the stream (programmatic dependent
//    launch); every wait is bounded (a timeout sets the error word);
//  * warps 0-7 consume, each owning 8 cells of every tile and its own online
//    softmax state, with no barrier between warps inside an item: scores with
//    four lanes per cell (32 of the 128 d each, fp16 K times fp32 Q in fp32
//    FMA, summed by two shuffles), softmax in base 2 (the running maximum is
//    moved only when it grows by more than 2^8), PV with each lane owning 4 of
//    the 128 d;
//  * cells outside the block's sequence are skipped in PV, so a NaN in an
//    unused cell cannot leak (masked cells of the sequence hold finite data);
//  * at an item's end the 8 warp states are merged in three rounds through
//    shared memory; a block covered by one item is written at once, the items
//    of a split block leave partials that the last CTA to finish merges
//    (atomic count, no spinning):
//      O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.

#include "dev_common.cuh"
#include "kernels.h"

namespace {

using kvi::TILE;
using kvi::DEC_QMAX;

constexpr int NW = 8;                           // consumer warps
constexpr int NCONS = NW * 32;
constexpr int NT = NCONS + 32;                  // + producer warp
constexpr int BOX_BYTES = TILE * 128;           // 64 rows x 64 fp16
constexpr int STAGE_BYTES = 4 * BOX_BYTES;      // K lo, K hi, V lo, V hi
constexpr int PART_STRIDE = 132;                // m, l, pad, pad, o[128]
constexpr float RESCALE_LOG2 = 8.0f;

template <int NQ>
constexpr int stages_for() { return NQ <= 4 ? 3 : 2; }

// A stage holds either one fully visible tile (64 cells, no per-cell test) or
// up to 8 packed 8-cell groups taken from the block's partially visible tiles,
// in the order the tile list gives them; slot w (cells 8w .. 8w + 7) belongs
// to consumer warp w.  The order of cells does not change the softmax.
struct Meta {                 // per stage: what the producer learned about its cells
    int32_t full;             // 1: one fully visible tile
    int32_t gmask;            // packed: bit w set when slot w holds a group
    int32_t last;             // the item's last stage
    int32_t pad;
    int32_t cpos[TILE];
    uint8_t has[TILE];        // cell holds the block's sequence and is not from a later ubatch
};

constexpr int GROUP_BYTES = 8 * 128;            // one 8-row box
constexpr int WINDOW = 32;                      // tile-list entries the producer reads at once
constexpr int GQ = 512;                         // group queue ring (> WINDOW * 8 + 7)

template <int NQ>
struct __align__(16) Aux {
    static constexpr int S = stages_for<NQ>();
    static constexpr int PQ = NQ < 4 ? 4 : NQ;  // padded for 16-byte loads
    Meta meta[S];
    float q[NQ][4][36];           // queries in fp32: q[n][dq][j] = Q[n][32 dq + j]
    float p[NW][8][PQ];           // each warp's probabilities, cell-major (NQ > 4)
    uint16_t ph[NW][8][4];        // ... as fp16 (NQ <= 4)
    float scr_m[4][NQ];           // tree merge: the writing warps' maxima,
    float scr_l[4][NQ];           //   row sums
    float scr_o[4][NQ][128];      //   and accumulators
    int32_t rpos[NQ];
    int32_t gq[GQ];               // producer: queued groups' first cells (in the stream)
    uint64_t full[S], empty[S];
    uint64_t cbar;                // consumer exchanges (all 256 consumer threads)
    int32_t fail;
    int32_t last_piece;           // this CTA completed the last piece of the item's block
};

template <int NQ>
constexpr size_t smem_bytes() { return (size_t)stages_for<NQ>() * STAGE_BYTES + sizeof(Aux<NQ>); }

// two CTAs per SM (228 KiB of shared memory, 1 KiB reserved per CTA) up to NQ = 8
static_assert(2 * (smem_bytes<4>() + 1024) <= 228 * 1024, "two NQ=4 CTAs must fit on an SM");
static_assert(2 * (smem_bytes<8>() + 1024) <= 228 * 1024, "two NQ=8 CTAs must fit on an SM");

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// d0 += a.lo * b.lo and d1 += a.hi * b.hi: a and b hold two fp16 each, the
// products are exact in fp32 and the sums are fp32 (one mixed-precision FMA each).
__device__ __forceinline__ void fma2_h(uint32_t a, uint32_t b, float &d0, float &d1) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\tfma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
        : "+f"(d0), "+f"(d1) : "r"(a), "r"(b));
}

// d[j] += p * v_j for the four fp16 v_j of two words (p fp16, sums fp32).
__device__ __forceinline__ void fma4_h(uint16_t p, uint32_t v01, uint32_t v23, float (&d)[4]) {
    asm("{\n\t.reg .b16 a0, a1, a2, a3;\n\t"
        "mov.b32 {a0, a1}, %5;\n\tmov.b32 {a2, a3}, %6;\n\t"
        "fma.rn.f32.f16 %0, %4, a0, %0;\n\tfma.rn.f32.f16 %1, %4, a1, %1;\n\t"
        "fma.rn.f32.f16 %2, %4, a2, %2;\n\tfma.rn.f32.f16 %3, %4, a3, %3;\n\t}"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3]) : "h"(p), "r"(v01), "r"(v23));
}

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

// All 256 consumer threads meet (arrive, then a bounded wait: a thread that
// gave up elsewhere makes the others time out instead of hanging).
__device__ __forceinline__ bool cons_sync(uint64_t *bar, uint32_t &phase, volatile int32_t *fail) {
    kvd::mbar_arrive(bar);
    const bool ok = __all_sync(0xffffffffu, wait_or_fail(bar, phase & 1u, fail));
    ++phase;
    return ok;
}

template <int NQ>
__global__ void __launch_bounds__(NT, (NQ <= 8 ? 2 : 1))
k_decode(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         const __grid_constant__ CUtensorMap tm_k8, const __grid_constant__ CUtensorMap tm_v8,
         const kvk::DecodeArgs a) {
    constexpr int S = stages_for<NQ>();
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *stages = smem;
    Aux<NQ> &x = *reinterpret_cast<Aux<NQ> *>(smem + (size_t)S * STAGE_BYTES);
    volatile int32_t *fail = &x.fail;
    const int32_t tid = threadIdx.x;
    const int32_t lane = tid & 31, warp = tid >> 5;
    const int32_t hk = blockIdx.y;
    const int32_t G = a.gqa;
    // Launched as a programmatic dependent: the plan, tables and cell mirror are
    // read before waiting for the previous kernel only when they were complete
    // before it began; Q, the K/V cache and the outputs only after the wait.
    if (!a.early_ok) kvd::pdl_wait();
    if (tid == 0) kvd::pdl_trigger();
    const int32_t i0 = a.p.cta_item0[blockIdx.x];
    const int32_t i1 = a.p.cta_item0[blockIdx.x + 1];

    if ((kvd::smem_u32(smem) & 1023u) != 0) {   // TMA swizzle needs 1 KiB alignment
        if (tid == 0) kvd::report(a.err, kvd::DERR_BOUNDS);
        return;
    }
    if (tid == 0) {
        kvd::prefetch_tmap(&tm_k);
        kvd::prefetch_tmap(&tm_v);
        kvd::prefetch_tmap(&tm_k8);
        kvd::prefetch_tmap(&tm_v8);
        for (int s = 0; s < S; ++s) {
            kvd::mbar_init(&x.full[s], 33);    // producer lane 0's expect_tx + 32 lanes
            kvd::mbar_init(&x.empty[s], NW);   // one arrival per consumer warp
        }
        kvd::mbar_init(&x.cbar, NCONS);
        x.fail = 0;
        kvd::fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ======================= producer =======================
        // Per item, the tile list is read WINDOW entries at a time: each fully
        // visible tile gets a stage of its own (four 64-row boxes); the visible
        // 8-cell groups of the other tiles are queued and leave in stages of 8
        // (four 8-row boxes each), the remainder with the item's last window.
        int32_t k = 0;
        bool dep_done = false;
        bool ok = true;
        uint32_t qh = 0, qt = 0;   // group queue head and tail (ring indices)
        // the column's start record: the first window's entries without the chain
        // item -> block -> list -> flags
        const int4 *rp = reinterpret_cast<const int4 *>(a.p.dec_first + kvk::DEC_FIRST * blockIdx.x);
        const int4 r_t = rp[0], r_fl = rp[1], r_w = rp[2], r_b = rp[3];
        // warm L2 with the column's first four tiles (K and V, both d halves; a
        // prefetch returns nothing) while the previous kernel may still be storing
        if (lane < 16) {
            const int32_t h = lane >> 2;
            const int32_t t = h == 0 ? r_t.x : h == 1 ? r_t.y : h == 2 ? r_t.z : r_t.w;
            if (t >= 0) kvd::tma_prefetch_2d((lane & 2) ? &tm_v : &tm_k, hk * 128 + 64 * (lane & 1), r_w.w + t * TILE);
        }
        // wait outcomes and the loop conditions are agreed by the whole warp, so a
        // failure never splits it in front of __syncwarp
        auto acquire = [&](int32_t st) -> bool {
            if (k >= S &&
                !__all_sync(0xffffffffu, wait_or_fail(&x.empty[st], (uint32_t)((k / S) - 1) & 1u, fail)))
                return false;
            if (!dep_done) {   // the K/V rows of this ubatch are written by the kernel before
                kvd::pdl_wait();
                dep_done = true;
            }
            return true;
        };
        for (int32_t wi = i0; wi < i1 && ok; ++wi) {
            const bool first = wi == i0;
            kvk::WorkItem w;
            int32_t ybase, n_rows, seq0;
            if (first) {   // from the start record
                w.block = r_w.x;
                w.t0 = r_w.y;
                w.t1 = r_w.z;
                ybase = r_w.w;
                n_rows = r_b.x;
                seq0 = r_b.y;
            } else {
                w = a.p.work[wi];
                const kvi::DevBlock b = a.u.blocks[w.block];
                ybase = b.stream * a.u.kv_size;
                n_rows = b.n_rows;
                seq0 = b.seq0;
            }
            const int32_t *list = a.p.tiles + (int64_t)w.block * a.p.tile_stride;
            const uint32_t *flg = a.p.flags + (int64_t)w.block * a.p.tile_stride;
            const int32_t xk = hk * 128;
            for (int32_t base = w.t0; base < w.t1 && ok; base += WINDOW) {
                const int32_t li = base + lane;
                int32_t t = 0;
                uint32_t fl = 0;
                if (li < w.t1) {
                    if (first && base == w.t0 && lane < 4) {
                        t = lane == 0 ? r_t.x : lane == 1 ? r_t.y : lane == 2 ? r_t.z : r_t.w;
                        fl = (uint32_t)(lane == 0 ? r_fl.x : lane == 1 ? r_fl.y : lane == 2 ? r_fl.z : r_fl.w);
                    } else {
                        t = list[li];
                        fl = flg[t];
                    }
                }
                const bool isfull = li < w.t1 && (int32_t)(fl & 0xffffu) == n_rows * TILE;
                uint32_t fm = __ballot_sync(0xffffffffu, isfull);
                // queue the visible groups of my tile (flags bits 16..23), in list order
                uint32_t gm = (li < w.t1 && !isfull) ? ((fl >> 16) & 0xffu) : 0u;
                const int32_t cnt = __popc(gm);
                int32_t incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                uint32_t pos = qt + (uint32_t)(incl - cnt);
                while (gm) {
                    const int32_t g = __ffs(gm) - 1;
                    gm &= gm - 1;
                    x.gq[pos++ & (GQ - 1)] = t * TILE + 8 * g;
                }
                qt += (uint32_t)__shfl_sync(0xffffffffu, incl, 31);
                __syncwarp();
                const bool final_window = base + WINDOW >= w.t1;
                // ---- fully visible tiles: one stage each ----
                while (fm && ok) {
                    const int32_t src = __ffs(fm) - 1;
                    fm &= fm - 1;
                    const int32_t tt = __shfl_sync(0xffffffffu, t, src);
                    const int32_t st = k % S;
                    if (!(ok = acquire(st))) break;
                    if (lane == 0) {
                        uint8_t *sp = stages + (size_t)st * STAGE_BYTES;
                        const int32_t y = ybase + tt * TILE;
                        x.meta[st].full = 1;
                        x.meta[st].gmask = 0xff;
                        x.meta[st].last = (final_window && fm == 0 && qt == qh) ? 1 : 0;
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive_expect_tx(&x.full[st], STAGE_BYTES);
                        kvd::tma_load_2d(sp, &tm_k, xk, y, &x.full[st]);
                        kvd::tma_load_2d(sp + BOX_BYTES, &tm_k, xk + 64, y, &x.full[st]);
                        kvd::tma_load_2d(sp + 2 * BOX_BYTES, &tm_v, xk, y, &x.full[st]);
                        kvd::tma_load_2d(sp + 3 * BOX_BYTES, &tm_v, xk + 64, y, &x.full[st]);
                    }
                    __syncwarp();
                    kvd::mbar_arrive(&x.full[st]);
                    ++k;
                }
                // ---- packed stages of 8 groups; the remainder on the item's last window ----
                while (ok && (qt - qh >= 8u || (final_window && qt != qh))) {
                    const int32_t n = (int32_t)min(8u, qt - qh);
                    const bool last = final_window && qt - qh <= 8u;
                    // the cells' visibility, read before the stage is free
                    bool hs[2] = {false, false};
                    int32_t cp[2] = {0, 0};
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int32_t l = lane + 32 * r;
                        if (l < 8 * n) {
                            const int32_t j = x.gq[(qh + (uint32_t)(l >> 3)) & (GQ - 1)] + (l & 7);
                            if (j < a.u.n_kv) {
                                const int64_t g = (int64_t)ybase + j;
                                const uint64_t wb = a.u.cell_bits[g * a.u.n_words + (seq0 >> 6)];
                                hs[r] = ((wb >> (seq0 & 63)) & 1ull) && a.u.cell_epoch[g] <= a.u.ub_epoch;
                                cp[r] = a.u.cell_pos[g];
                            }
                        }
                    }
                    const int32_t jg = lane < n ? x.gq[(qh + (uint32_t)lane) & (GQ - 1)] : 0;
                    const int32_t st = k % S;
                    if (!(ok = acquire(st))) break;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        x.meta[st].has[lane + 32 * r] = hs[r] ? 1 : 0;
                        x.meta[st].cpos[lane + 32 * r] = cp[r];
                    }
                    if (lane == 0) {
                        x.meta[st].full = 0;
                        x.meta[st].gmask = (1 << n) - 1;
                        x.meta[st].last = last ? 1 : 0;
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive_expect_tx(&x.full[st], (uint32_t)(n * 4 * GROUP_BYTES));
                    }
                    __syncwarp();
                    if (lane < n) {   // slot `lane` of the stage: rows jg .. jg + 7
                        uint8_t *sp = stages + (size_t)st * STAGE_BYTES + lane * GROUP_BYTES;
                        const int32_t y = ybase + jg;
                        kvd::tma_load_2d(sp, &tm_k8, xk, y, &x.full[st]);
                        kvd::tma_load_2d(sp + BOX_BYTES, &tm_k8, xk + 64, y, &x.full[st]);
                        kvd::tma_load_2d(sp + 2 * BOX_BYTES, &tm_v8, xk, y, &x.full[st]);
                        kvd::tma_load_2d(sp + 3 * BOX_BYTES, &tm_v8, xk + 64, y, &x.full[st]);
                    }
                    qh += (uint32_t)n;
                    __syncwarp();
                    kvd::mbar_arrive(&x.full[st]);
                    ++k;
                }
            }
        }
        if (*fail && lane == 0) {
            // let copies already in flight land before the CTA's smem is released
            for (int32_t q = k > S ? k - S : 0; q < k; ++q)
                (void)kvd::mbar_wait_bounded(&x.full[q % S], (uint32_t)(q / S) & 1u);
        }
    } else {
        // ======================= consumers =======================
        const int32_t c = lane >> 2;               // scores: my cell among the warp's 8
        const int32_t dq = lane & 3;               // scores: my quarter of d
        const int32_t cw = warp * 8 + c;           // my cell within the tile
        uint32_t cph = 0;                          // consumer-barrier phase
        int32_t k = 0;
        bool ok = true;
        bool dep_done = false;
        for (int32_t wi = i0; wi < i1 && ok; ++wi) {
            const kvk::WorkItem w = a.p.work[wi];
            const kvi::DevBlock b = a.u.blocks[w.block];
            const int32_t nq = b.n_rows * G;
            if (!dep_done) {   // before the first read of Q and the first write of an output
                kvd::pdl_wait();
                dep_done = true;
            }
            // NQ <= 4: my 16 of the 128 d of every query vector (d = 8e .. 8e + 7 and
            // 64 + 8e .. 64 + 8e + 7), fp16, stay in registers for the whole item
            constexpr bool RQ = NQ <= 4;
            const int32_t g = lane >> 3, e = lane & 7;
            uint32_t qh[NQ][8];
            int32_t rp[NQ];
            if constexpr (RQ) {
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                    rp[n] = 0;
                    if (n < nq) {
                        const int32_t row = a.u.perm[b.row0 + n / G];
                        const int32_t h = hk * G + (n % G);
                        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((int64_t)row * a.n_head + h) * 128);
                        lo = src[e];
                        hi = src[8 + e];
                        rp[n] = a.u.rows[row].pos;
                    }
                    qh[n][0] = lo.x; qh[n][1] = lo.y; qh[n][2] = lo.z; qh[n][3] = lo.w;
                    qh[n][4] = hi.x; qh[n][5] = hi.y; qh[n][6] = hi.z; qh[n][7] = hi.w;
                }
            } else {   // ---- NQ > 4: Q (fp32) and the rows' positions in shared memory ----
                const int32_t n = tid >> 4, part = tid & 15;   // 8 values of query vector n
                if (n < NQ) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0.f;
                    if (n < nq) {
                        const int32_t row = a.u.perm[b.row0 + n / G];
                        const int32_t h = hk * G + (n % G);
                        const uint4 raw =
                            *reinterpret_cast<const uint4 *>(a.q + ((int64_t)row * a.n_head + h) * 128 + 8 * part);
                        const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(h2[e]);
                            v[2 * e] = f.x;
                            v[2 * e + 1] = f.y;
                        }
                    }
                    float *dst = &x.q[n][part >> 2][(part & 3) * 8];
                    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<float4 *>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
                }
                if (tid < NQ) x.rpos[tid] = tid < nq ? a.u.rows[a.u.perm[b.row0 + tid / G]].pos : 0;
                if (!(ok = cons_sync(&x.cbar, cph, fail))) break;
            }

            float m[NQ], lp[NQ], acc[NQ][4];
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                m[n] = -INFINITY;
                lp[n] = 0.f;
                acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
            }
            // NQ == 4: after the score reduction each lane holds one query vector,
            // nl = (e >> 1) & 3, with its own running maximum and row-sum part
            const int32_t nl = (e >> 1) & 3;
            float m_l = -INFINITY, lp_l = 0.f;
            int32_t rp_l = 0;
            if constexpr (NQ == 4) {
#pragma unroll
                for (int n = 0; n < NQ; ++n)
                    if (nl == n) rp_l = rp[n];
            }
            // the item's stages, until the one marked last (an item with an empty
            // list has none)
            for (bool more = w.t0 < w.t1; more; ++k) {
                const int32_t st = k % S;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.full[st], (uint32_t)(k / S) & 1u, fail));
                if (!ok) break;
                const uint8_t *sp = stages + (size_t)st * STAGE_BYTES;
                const bool full = x.meta[st].full != 0;
                more = x.meta[st].last == 0;
                if (!((x.meta[st].gmask >> warp) & 1)) {   // my slot of a packed stage is empty
                    __syncwarp();
                    if (lane == 0) kvd::mbar_arrive(&x.empty[st]);
                    continue;
                }
                if constexpr (NQ == 4) {
                // ---- scores: cells g and g + 4 of my warp's 8, my 16 d, the four query
                //      vectors; the eight lanes of a cell then reduce-scatter the sums so
                //      that lane e keeps query nl (4 shuffles instead of 12) ----
                const int32_t c0 = warp * 8 + g, c1 = c0 + 4;
                float scv[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int32_t cell = r ? c1 : c0;
                    const uint4 k0 = *reinterpret_cast<const uint4 *>(sp + kvd::swz128(cell, e));
                    const uint4 k1 = *reinterpret_cast<const uint4 *>(sp + BOX_BYTES + kvd::swz128(cell, e));
                    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                    float dd[4];
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) fma2_h(kw[j], qh[n][j], d0, d1);
                        dd[n] = d0 + d1;
                    }
                    const bool up = (e & 4) != 0;       // lanes e >= 4 keep queries 2, 3
                    float ka = up ? dd[2] : dd[0], kb = up ? dd[3] : dd[1];
                    const float sa = up ? dd[0] : dd[2], sb = up ? dd[1] : dd[3];
                    ka += __shfl_xor_sync(0xffffffffu, sa, 4);
                    kb += __shfl_xor_sync(0xffffffffu, sb, 4);
                    const bool up2 = (e & 2) != 0;      // then the second of the pair
                    float kv = up2 ? kb : ka;
                    kv += __shfl_xor_sync(0xffffffffu, up2 ? ka : kb, 2);
                    kv += __shfl_xor_sync(0xffffffffu, kv, 1);
                    scv[r] = kv;
                }
                const bool h0 = full || x.meta[st].has[c0], h1 = full || x.meta[st].has[c1];
                const int32_t p0 = full ? 0 : x.meta[st].cpos[c0], p1 = full ? 0 : x.meta[st].cpos[c1];
                const bool v0 = h0 && nl < nq && (full || kvd::pos_visible(a.u.causal, a.u.n_swa, rp_l, p0));
                const bool v1 = h1 && nl < nq && (full || kvd::pos_visible(a.u.causal, a.u.n_swa, rp_l, p1));
                const float s0 = v0 ? scv[0] * a.scale_log2 : -INFINITY;
                const float s1 = v1 ? scv[1] * a.scale_log2 : -INFINITY;
                // ---- online softmax of query nl over my warp's 8 cells ----
                float t = fmaxf(s0, s1);
                t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
                t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
                const float mn = fmaxf(m_l, t);
                const bool grow = mn > m_l + RESCALE_LOG2 || (m_l == -INFINITY && mn != -INFINITY);
                float al = 1.f;
                if (grow) {
                    al = ex2_approx(m_l - mn);
                    m_l = mn;
                    lp_l *= al;
                }
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int n = 0; n < 4; ++n) {   // lane 2n holds query n
                        const float an = __shfl_sync(0xffffffffu, al, 2 * n);
                        acc[n][0] *= an;
                        acc[n][1] *= an;
                        acc[n][2] *= an;
                        acc[n][3] *= an;
                    }
                }
                {
                    const bool live = m_l != -INFINITY;
                    const __half q0 = __float2half_rn(live ? ex2_approx(s0 - m_l) : 0.f);
                    const __half q1 = __float2half_rn(live ? ex2_approx(s1 - m_l) : 0.f);
                    if ((e & 1) == 0) {   // the row sum counts P as the PV product sees it (fp16)
                        lp_l += __half2float(q0) + __half2float(q1);
                        x.ph[warp][g][nl] = __half_as_ushort(q0);
                        x.ph[warp][g + 4][nl] = __half_as_ushort(q1);
                    }
                }
                __syncwarp();
                // ---- O += P V over my warp's 8 cells; lane owns d = 4 lane .. 4 lane + 3 ----
                {
                    const uint8_t *vb = sp + 2 * BOX_BYTES + (lane >> 4) * BOX_BYTES;
                    const uint32_t chunk = (uint32_t)(lane & 15) >> 1, inner = (uint32_t)(lane & 1) * 8u;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int32_t cell = warp * 8 + cc;
                        if (!full && !x.meta[st].has[cell]) continue;   // warp-uniform
                        const uint2 raw = *reinterpret_cast<const uint2 *>(vb + kvd::swz128(cell, chunk) + inner);
                        const uint2 pw = *reinterpret_cast<const uint2 *>(&x.ph[warp][cc][0]);
                        fma4_h((uint16_t)(pw.x & 0xffffu), raw.x, raw.y, acc[0]);
                        fma4_h((uint16_t)(pw.x >> 16), raw.x, raw.y, acc[1]);
                        fma4_h((uint16_t)(pw.y & 0xffffu), raw.x, raw.y, acc[2]);
                        fma4_h((uint16_t)(pw.y >> 16), raw.x, raw.y, acc[3]);
                    }
                }
                } else if constexpr (RQ) {
                // ---- scores: cells g and g + 4 of my warp's 8, my 16 d, all query vectors
                //      (fp16 K times fp16 Q, fp32 sums; eight lanes per cell) ----
                const int32_t c0 = warp * 8 + g, c1 = c0 + 4;
                float sc[2][NQ];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int32_t cell = r ? c1 : c0;
                    const uint4 k0 = *reinterpret_cast<const uint4 *>(sp + kvd::swz128(cell, e));
                    const uint4 k1 = *reinterpret_cast<const uint4 *>(sp + BOX_BYTES + kvd::swz128(cell, e));
                    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int j = 0; j < 8; ++j) fma2_h(kw[j], qh[n][j], d0, d1);
                        float v = d0 + d1;
                        v += __shfl_xor_sync(0xffffffffu, v, 1);
                        v += __shfl_xor_sync(0xffffffffu, v, 2);
                        v += __shfl_xor_sync(0xffffffffu, v, 4);
                        sc[r][n] = v;
                    }
                }
                const bool h0 = full || x.meta[st].has[c0], h1 = full || x.meta[st].has[c1];
                const int32_t p0 = full ? 0 : x.meta[st].cpos[c0], p1 = full ? 0 : x.meta[st].cpos[c1];
                // ---- online softmax over my warp's 8 cells (warp-uniform decisions) ----
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    const bool v0 = h0 && n < nq && (full || kvd::pos_visible(a.u.causal, a.u.n_swa, rp[n], p0));
                    const bool v1 = h1 && n < nq && (full || kvd::pos_visible(a.u.causal, a.u.n_swa, rp[n], p1));
                    const float s0 = v0 ? sc[0][n] * a.scale_log2 : -INFINITY;
                    const float s1 = v1 ? sc[1][n] * a.scale_log2 : -INFINITY;
                    float t = fmaxf(s0, s1);
                    t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
                    t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
                    const float mn = fmaxf(m[n], t);
                    if (mn > m[n] + RESCALE_LOG2 || (m[n] == -INFINITY && mn != -INFINITY)) {
                        const float al = ex2_approx(m[n] - mn);
                        lp[n] *= al;
                        acc[n][0] *= al;
                        acc[n][1] *= al;
                        acc[n][2] *= al;
                        acc[n][3] *= al;
                        m[n] = mn;
                    }
                    const bool live = m[n] != -INFINITY;
                    const __half q0 = __float2half_rn(live ? ex2_approx(s0 - m[n]) : 0.f);
                    const __half q1 = __float2half_rn(live ? ex2_approx(s1 - m[n]) : 0.f);
                    if (e == 0) {   // the row sum counts P as the PV product sees it (fp16)
                        lp[n] += __half2float(q0) + __half2float(q1);
                        x.ph[warp][g][n] = __half_as_ushort(q0);
                        x.ph[warp][g + 4][n] = __half_as_ushort(q1);
                    }
                }
                __syncwarp();
                // ---- O += P V over my warp's 8 cells; lane owns d = 4 lane .. 4 lane + 3 ----
                {
                    const uint8_t *vb = sp + 2 * BOX_BYTES + (lane >> 4) * BOX_BYTES;
                    const uint32_t chunk = (uint32_t)(lane & 15) >> 1, inner = (uint32_t)(lane & 1) * 8u;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int32_t cell = warp * 8 + cc;
                        if (!full && !x.meta[st].has[cell]) continue;   // warp-uniform
                        const uint2 raw = *reinterpret_cast<const uint2 *>(vb + kvd::swz128(cell, chunk) + inner);
                        const uint2 pw = *reinterpret_cast<const uint2 *>(&x.ph[warp][cc][0]);
                        const uint16_t pq[4] = {(uint16_t)(pw.x & 0xffffu), (uint16_t)(pw.x >> 16),
                                                (uint16_t)(pw.y & 0xffffu), (uint16_t)(pw.y >> 16)};
#pragma unroll
                        for (int n = 0; n < NQ; ++n) fma4_h(pq[n], raw.x, raw.y, acc[n]);
                    }
                }
                } else {
                // ---- scores: my cell, my 32 d, all query vectors ----
                float s[NQ];
#pragma unroll
                for (int n = 0; n < NQ; ++n) s[n] = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ch = 4 * dq + i;             // 16-byte chunk of the 256-byte K row
                    const uint4 raw =
                        *reinterpret_cast<const uint4 *>(sp + (ch >> 3) * BOX_BYTES + kvd::swz128(cw, ch & 7));
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
                    float kf[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(h2[e]);
                        kf[2 * e] = f.x;
                        kf[2 * e + 1] = f.y;
                    }
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        const float4 qa = *reinterpret_cast<const float4 *>(&x.q[n][dq][8 * i]);
                        const float4 qb = *reinterpret_cast<const float4 *>(&x.q[n][dq][8 * i + 4]);
                        float d0 = s[n];
                        d0 = fmaf(qa.x, kf[0], d0);
                        d0 = fmaf(qa.y, kf[1], d0);
                        d0 = fmaf(qa.z, kf[2], d0);
                        d0 = fmaf(qa.w, kf[3], d0);
                        d0 = fmaf(qb.x, kf[4], d0);
                        d0 = fmaf(qb.y, kf[5], d0);
                        d0 = fmaf(qb.z, kf[6], d0);
                        d0 = fmaf(qb.w, kf[7], d0);
                        s[n] = d0;
                    }
                }
                const bool has = full || x.meta[st].has[cw];
                const int32_t cpos = full ? 0 : x.meta[st].cpos[cw];
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    float v = s[n];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    const bool vis = has && n < nq && (full || kvd::pos_visible(a.u.causal, a.u.n_swa, x.rpos[n], cpos));
                    s[n] = vis ? v * a.scale_log2 : -INFINITY;
                }
                // ---- online softmax over my warp's 8 cells (warp-uniform decisions) ----
#pragma unroll
                for (int n = 0; n < NQ; ++n) {
                    float t = s[n];
                    t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 4));
                    t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
                    t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
                    const float mn = fmaxf(m[n], t);
                    if (mn > m[n] + RESCALE_LOG2 || (m[n] == -INFINITY && mn != -INFINITY)) {
                        const float al = ex2_approx(m[n] - mn);
                        lp[n] *= al;
                        acc[n][0] *= al;
                        acc[n][1] *= al;
                        acc[n][2] *= al;
                        acc[n][3] *= al;
                        m[n] = mn;
                    }
                    const float pv = m[n] == -INFINITY ? 0.f : ex2_approx(s[n] - m[n]);
                    if (dq == 0) {
                        lp[n] += pv;
                        x.p[warp][c][n] = pv;
                    }
                }
                __syncwarp();
                // ---- O += P V over my warp's 8 cells; lane owns d = 4 lane .. 4 lane + 3 ----
                {
                    const uint8_t *vb = sp + 2 * BOX_BYTES + (lane >> 4) * BOX_BYTES;
                    const uint32_t chunk = (uint32_t)(lane & 15) >> 1, inner = (uint32_t)(lane & 1) * 8u;
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const int32_t cell = warp * 8 + cc;
                        if (!full && !x.meta[st].has[cell]) continue;   // warp-uniform
                        const uint2 raw = *reinterpret_cast<const uint2 *>(vb + kvd::swz128(cell, chunk) + inner);
                        const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
                        const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
#pragma unroll
                        for (int n4 = 0; n4 < NQ; n4 += 4) {
                            const float4 pp = *reinterpret_cast<const float4 *>(&x.p[warp][cc][n4]);
                            const float pq[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (n4 + e < NQ) {
                                    acc[n4 + e][0] = fmaf(pq[e], v01.x, acc[n4 + e][0]);
                                    acc[n4 + e][1] = fmaf(pq[e], v01.y, acc[n4 + e][1]);
                                    acc[n4 + e][2] = fmaf(pq[e], v23.x, acc[n4 + e][2]);
                                    acc[n4 + e][3] = fmaf(pq[e], v23.y, acc[n4 + e][3]);
                                }
                            }
                        }
                    }
                }
                }   // NQ > 4
                __syncwarp();
                if (lane == 0) kvd::mbar_arrive(&x.empty[st]);   // release the stage (K, V, metadata)
            }
            if (!ok) break;

            // ---- the item's result: merge the 8 warps (three rounds) ----
            if constexpr (NQ == 4) {   // back to one (m, l part) per query vector on every lane
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    m[n] = __shfl_sync(0xffffffffu, m_l, 2 * n);
                    lp[n] = (nl == n && (e & 1) == 0) ? lp_l : 0.f;
                }
            }
            float l[NQ];
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                float v = lp[n];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                l[n] = v;
            }
            // Three rounds, one exchange each: in round sd, warp sd + j writes slot
            // (sd == 4 ? j : sd + j) and warp j merges it.  A slot is written again only
            // by the warp that read it in the round before, so no second exchange is
            // needed between rounds; one more after the last round keeps the next
            // item's writers off slot 1 until warp 0 has read it.
            for (int sd = 4; sd >= 1 && ok; sd >>= 1) {
                if (warp >= sd && warp < 2 * sd) {
                    const int slot = sd == 4 ? warp - sd : warp;
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        if (lane == 0) {
                            x.scr_m[slot][n] = m[n];
                            x.scr_l[slot][n] = l[n];
                        }
                        *reinterpret_cast<float4 *>(&x.scr_o[slot][n][4 * lane]) =
                            make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
                    }
                }
                if (!(ok = cons_sync(&x.cbar, cph, fail))) break;
                if (warp < sd) {
                    const int slot = sd == 4 ? warp : sd + warp;
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        const float m2 = x.scr_m[slot][n], l2 = x.scr_l[slot][n];
                        const float4 o2 = *reinterpret_cast<const float4 *>(&x.scr_o[slot][n][4 * lane]);
                        const float mn = fmaxf(m[n], m2);
                        const float a1 = m[n] == -INFINITY ? 0.f : ex2_approx(m[n] - mn);
                        const float a2 = m2 == -INFINITY ? 0.f : ex2_approx(m2 - mn);
                        l[n] = l[n] * a1 + l2 * a2;
                        acc[n][0] = acc[n][0] * a1 + o2.x * a2;
                        acc[n][1] = acc[n][1] * a1 + o2.y * a2;
                        acc[n][2] = acc[n][2] * a1 + o2.z * a2;
                        acc[n][3] = acc[n][3] * a1 + o2.w * a2;
                        m[n] = mn;
                    }
                }
            }
            if (ok) ok = cons_sync(&x.cbar, cph, fail);
            if (!ok) break;
            if (warp == 0) {
                const int32_t nitems = a.p.blk_nitems[w.block];
                if (nitems == 1) {
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        if (n < nq) {
                            const float inv = l[n] > 0.f ? 1.f / l[n] : 0.f;
                            const int32_t row = a.u.perm[b.row0 + n / G];
                            const int32_t h = hk * G + (n % G);
                            *reinterpret_cast<float4 *>(a.o + ((int64_t)row * a.n_head + h) * 128 + 4 * lane) =
                                make_float4(acc[n][0] * inv, acc[n][1] * inv, acc[n][2] * inv, acc[n][3] * inv);
                        }
                    }
                } else {
                    float *pp = a.part + ((int64_t)wi * a.n_head_kv + hk) * DEC_QMAX * PART_STRIDE;
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        if (n < nq) {
                            if (lane == 0) {
                                pp[n * PART_STRIDE + 0] = m[n];
                                pp[n * PART_STRIDE + 1] = l[n];
                            }
                            *reinterpret_cast<float4 *>(pp + n * PART_STRIDE + 4 + 4 * lane) =
                                make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
                        }
                    }
                    // the warp's partial writes come before lane 0's count, which
                    // releases them (and, for the last piece, acquires the others')
                    __syncwarp();
                    int32_t prev = 0;
                    if (lane == 0)
                        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                                     : "=r"(prev) : "l"(&a.p.counters[w.block * a.n_head_kv + hk]) : "memory");
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    if (lane == 0) x.last_piece = prev == nitems - 1 ? 1 : 0;
                }
            }
            // A split block: the CTA that completed its last piece merges every piece's
            // partial with all eight warps:
            //   O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q.
            // Each query vector gets wpn warps, each warp every wpn-th piece: its lanes
            // read the pieces' (m, l) together and each lane owns 4 of the 128 d of O,
            // the first O rows loaded alongside (m, l); a warp keeps a running maximum
            // across rounds of 32 pieces.  The wpn warp states of a query vector then
            // meet in the tree-merge scratch (room for 4 NQ states).
            const int32_t nitems_b = a.p.blk_nitems[w.block];
            if (nitems_b > 1) {
                if (!(ok = cons_sync(&x.cbar, cph, fail))) break;
                if (x.last_piece) {
                    // (warp 0's acquiring count came before the exchange above)
                    const int32_t it0 = a.p.blk_item0[w.block];
                    const int64_t istride = (int64_t)a.n_head_kv * DEC_QMAX * PART_STRIDE;
                    const float *pb = a.part + ((int64_t)it0 * a.n_head_kv + hk) * DEC_QMAX * PART_STRIDE;
                    const int32_t wpn = max(1, min(NW, 4 * NQ) / nq);   // warps per query vector
                    const int32_t sub = warp % wpn;
                    const int32_t myc = (nitems_b - sub + wpn - 1) / wpn;   // my pieces: sub + wpn j
                    float *sm = &x.scr_m[0][0], *sl = &x.scr_l[0][0], *so = &x.scr_o[0][0][0];
                    for (int32_t n = warp / wpn; n < nq; n += NW / wpn) {
                        const float *pn = pb + n * PART_STRIDE;
                        auto orow = [&](int32_t j) -> float4 {
                            return __ldcg(reinterpret_cast<const float4 *>(pn + (int64_t)(sub + wpn * j) * istride + 4) + lane);
                        };
                        float Mw = -INFINITY, Lw = 0.f;
                        float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int32_t j0 = 0; j0 < myc; j0 += 32) {
                            const int32_t nb = min(32, myc - j0);
                            float4 ov[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) ov[u] = u < nb ? orow(j0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
                            float mq = -INFINITY, lq = 0.f;
                            if (lane < nb) {
                                const float *pq = pn + (int64_t)(sub + wpn * (j0 + lane)) * istride;
                                mq = __ldcg(pq);
                                lq = __ldcg(pq + 1);
                            }
                            float Mc = mq;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, o));
                            const float Mn = fmaxf(Mw, Mc);
                            const float rs = Mw == -INFINITY ? 0.f : ex2_approx(Mw - Mn);
                            const float sq = mq == -INFINITY ? 0.f : ex2_approx(mq - Mn);
                            float lsum = lq * sq;
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
                            Lw = Lw * rs + lsum;
                            o4.x *= rs;
                            o4.y *= rs;
                            o4.z *= rs;
                            o4.w *= rs;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float sc = __shfl_sync(0xffffffffu, sq, u);
                                o4.x = fmaf(ov[u].x, sc, o4.x);
                                o4.y = fmaf(ov[u].y, sc, o4.y);
                                o4.z = fmaf(ov[u].z, sc, o4.z);
                                o4.w = fmaf(ov[u].w, sc, o4.w);
                            }
#pragma unroll 4
                            for (int32_t qq = 4; qq < nb; ++qq) {
                                const float sc = __shfl_sync(0xffffffffu, sq, qq);
                                const float4 v = orow(j0 + qq);
                                o4.x = fmaf(v.x, sc, o4.x);
                                o4.y = fmaf(v.y, sc, o4.y);
                                o4.z = fmaf(v.z, sc, o4.z);
                                o4.w = fmaf(v.w, sc, o4.w);
                            }
                            Mw = Mn;
                        }
                        if (wpn == 1) {
                            const float inv = Lw > 0.f ? 1.f / Lw : 0.f;
                            const int32_t row = a.u.perm[b.row0 + n / G];
                            const int32_t h = hk * G + (n % G);
                            *reinterpret_cast<float4 *>(a.o + ((int64_t)row * a.n_head + h) * 128 + 4 * lane) =
                                make_float4(o4.x * inv, o4.y * inv, o4.z * inv, o4.w * inv);
                        } else {
                            const int32_t slot = n * wpn + sub;   // < nq wpn <= 4 NQ
                            if (lane == 0) {
                                sm[slot] = Mw;
                                sl[slot] = Lw;
                            }
                            *reinterpret_cast<float4 *>(so + slot * 128 + 4 * lane) = o4;
                        }
                    }
                    if (wpn > 1) {
                        if (!(ok = cons_sync(&x.cbar, cph, fail))) break;
                        if (sub == 0 && warp / wpn < nq) {
                            const int32_t n = warp / wpn;
                            float M = -INFINITY;
                            for (int32_t s2 = 0; s2 < wpn; ++s2) M = fmaxf(M, sm[n * wpn + s2]);
                            float L = 0.f;
                            float4 o4 = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (M != -INFINITY) {
                                for (int32_t s2 = 0; s2 < wpn; ++s2) {
                                    const int32_t slot = n * wpn + s2;
                                    const float ms = sm[slot];
                                    const float sc = ms == -INFINITY ? 0.f : ex2_approx(ms - M);
                                    const float4 v = *reinterpret_cast<const float4 *>(so + slot * 128 + 4 * lane);
                                    L = fmaf(sl[slot], sc, L);
                                    o4.x = fmaf(v.x, sc, o4.x);
                                    o4.y = fmaf(v.y, sc, o4.y);
                                    o4.z = fmaf(v.z, sc, o4.z);
                                    o4.w = fmaf(v.w, sc, o4.w);
                                }
                            }
                            const float inv = L > 0.f ? 1.f / L : 0.f;
                            const int32_t row = a.u.perm[b.row0 + n / G];
                            const int32_t h = hk * G + (n % G);
                            *reinterpret_cast<float4 *>(a.o + ((int64_t)row * a.n_head + h) * 128 + 4 * lane) =
                                make_float4(o4.x * inv, o4.y * inv, o4.z * inv, o4.w * inv);
                        }
                        // the next item's tree merge reuses the scratch
                        if (!(ok = cons_sync(&x.cbar, cph, fail))) break;
                    }
                    if (tid == 0) a.p.counters[w.block * a.n_head_kv + hk] = 0;   // for the next launch
                }
            }
        }
    }
    __syncthreads();
    if (*fail && tid == 0) kvd::report(a.err, kvd::DERR_TMA_TIMEOUT);
}

template <int NQ>
cudaError_t load_nq() {
    return cudaFuncSetAttribute(k_decode<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<NQ>());
}

// The shared-memory attribute was set for the current device by load_decode_kernels.
template <int NQ>
cudaError_t launch_nq(const CUtensorMap *tm, const kvk::DecodeArgs &a, int32_t grid_x, cudaStream_t st) {
    constexpr size_t SMEM = smem_bytes<NQ>();
    // a programmatic dependent of the kernel before it (normally the K/V store)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, a.n_head_kv);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_decode<NQ>, tm[0], tm[1], tm[2], tm[3], a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

namespace kvk {

int32_t decode_ctas_per_sm() { return 2; }

cudaError_t load_decode_kernels() {
    cudaError_t e;
    if ((e = load_nq<1>()) != cudaSuccess || (e = load_nq<2>()) != cudaSuccess || (e = load_nq<4>()) != cudaSuccess ||
        (e = load_nq<8>()) != cudaSuccess || (e = load_nq<16>()) != cudaSuccess)
        return e;
    return cudaSuccess;
}

cudaError_t launch_decode(const CUtensorMap *tm, const DecodeArgs &a, int32_t grid_x, cudaStream_t st) {
    if (a.nq_max <= 1) return launch_nq<1>(tm, a, grid_x, st);
    if (a.nq_max <= 2) return launch_nq<2>(tm, a, grid_x, st);
    if (a.nq_max <= 4) return launch_nq<4>(tm, a, grid_x, st);
    if (a.nq_max <= 8) return launch_nq<8>(tm, a, grid_x, st);
    return launch_nq<16>(tm, a, grid_x, st);
}

}  // namespace kvk
