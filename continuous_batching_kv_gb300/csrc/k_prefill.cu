// K3b: GQA flash attention, prefill / mixed path, on tcgen05 tensor cores.
//
// "llama.cpp and the ubatch", "Chunked prefill is the same mechanism": a
// chunk of U rows against C cached cells is a [U, C+U] score matrix; with the
// mask of "The mask is doing the work" (occupied, same first sequence id,
// not later) it is the same softmax(q K^T / sqrt(d) + mask) V as decode, but
// now a dense contraction worth putting on the tensor cores.
//
// Design (sm_103a, one CTA of 608 threads per SM):
//  * a block = up to 128 query vectors (rows sharing a stream and first
//    sequence id, times the GQA group) = the 128 TMEM lanes of one MMA tile;
//    a work item = one block, one KV head, a chunk of the block's list of
//    visible 64-cell tiles, consumed two at a time (N = 128 cells);
//  * warp 16 streams K tiles with TMA (128-byte swizzle) into a 3-slot ring,
//    with each pair's list entries, flags and per-cell visibility fetched ahead
//    into a metadata ring; warp 18 streams V tiles into a 3-slot ring; warp 17
//    allocates TMEM and one of its threads issues tcgen05.mma in a fixed order
//    (S_0, S_1, then PV_j and S_j+2 per pair, each after a blocking bounded
//    wait): S = Q K^T (M 128, N 128, K 128; Q held in TMEM) into one of two
//    TMEM score buffers, and O += P V with P read from TMEM (fp16, written over
//    S) and V MN-major from shared memory; tcgen05.commit signals the mbarriers;
//  * warps 0-15: thread (n, qd) owns cells 32qd .. 32qd + 31 of query vector n
//    (TMEM lane n) and d = 32qd .. 32qd + 31 of O; it reads its 32 columns of S
//    with one tcgen05.ld, applies the mask per cell on tiles that are not fully
//    visible, exchanges the row maximum with the row's other three threads,
//    runs the online softmax in base 2 (the exponent rounded to fp16, two
//    exponentials per ex2.approx.f16x2), writes P (fp16, two cells per 32-bit
//    column) at the start of the S columns it read, and rescales its part of O
//    in TMEM only when the running maximum grew by more than 2^8 (otherwise the
//    stale maximum is kept; the final normalisation uses the same one);
//  * cells nobody in the block may see get their V rows zeroed in shared
//    memory before the PV product (P is 0 there, but 0 * NaN would not be);
//  * a block split over several CTAs leaves one partial (m, l, O) per piece,
//    merged by a small second kernel launched as a programmatic dependent (it
//    reads the plan while this kernel runs); every mbarrier wait is bounded.

#include "dev_common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace {

using kvi::TILE;

constexpr int NSM = 512;                 // softmax threads: four per TMEM lane
constexpr int NT = NSM + 96;             // + K producer, MMA and V producer warps
constexpr int W_K = NSM / 32;            // K producer warp
constexpr int W_MMA = W_K + 1;           // TMEM allocation and MMA issue
constexpr int W_V = W_K + 2;             // V producer warp
constexpr int M = 128;
constexpr int HALF = 128 * 128;          // [128 rows][64 fp16], 128-byte rows
constexpr int TILEB = 2 * HALF;          // 32 KiB
constexpr int BOX = 64 * 128;            // one TMA box: 64 rows x 64 fp16
constexpr int KSTAGES = 3;             // K ring: K of pair g + 3 loads once S of g has read K of g
constexpr int VSTAGES = 3;             // V ring: V of pair g + 3 loads once PV of g is done
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KSTAGES * TILEB;
constexpr int OFF_AUX = OFF_V + VSTAGES * TILEB;
constexpr int PART_STRIDE = 132;
constexpr uint32_t TMEM_COLS = 512;      // S0 [0,128), S1 [128,256) (P written over S), O [256,384), Q [384,448)
constexpr uint32_t COL_O = 256;          // O: fp32 accumulator, d = 0 .. 127
constexpr uint32_t COL_Q = 384;          // Q: fp16, two d per column (the A operand of S = Q K^T)
constexpr float RESCALE_LOG2 = 8.0f;
constexpr unsigned POLL_NS = 32;         // back-off of the polling producer / MMA loops

constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16(128, 128, 0, 1);

// Metadata ring.  Pair g's slot is rewritten by the K load of pair g + MSLOTS,
// which needs S of g + MSLOTS - KSTAGES to be done, which was issued only after
// the PV of the pair before it in its score buffer (g + MSLOTS - KSTAGES - 2 or
// later) was issued, i.e. after the softmax finished that pair: with MSLOTS >=
// KSTAGES + 2 the softmax is done with pair g, and the V load of g (which reads
// the slot) went out before that PV.
constexpr int MSLOTS = 8;
static_assert(MSLOTS >= KSTAGES + 2, "metadata ring too short for the K ring");

struct __align__(16) Meta {     // per pair tile: what the producer learned about it (16-byte loads)
    int32_t full;
    int32_t ys[2];            // TMA row coordinates of the two 64-cell halves
    int32_t pad;
    int32_t cpos[128];
    uint8_t has[128];         // cell holds the block's sequence and is not from a later ubatch
    uint8_t anyvis[128];      // ... and some row of the block may see it
};

struct __align__(16) Aux {
    uint64_t k_full[KSTAGES], k_empty[KSTAGES], v_full[VSTAGES], v_empty[VSTAGES];
    uint64_t meta_full[MSLOTS];
    uint64_t s_full[2], p_full[2], pv_done[2], q_full, spare;   // p_full, pv_done [g & 1]: pair g
    uint64_t lbar;            // the halves' row-sum exchange at each item's end, all 256 threads
    uint64_t pbar[4];         // per lane quarter: the four warps of a row exchange maxima per pair
    uint32_t tmem_base;
    int32_t fail;
    int32_t flag;
    int32_t pad;
    Meta meta[MSLOTS];
    float red[2][4][M];       // [pair parity][cell quarter][row]: partial row maxima
    float lex[2][4][M];       // [item parity][cell quarter][row]: row sums
};

constexpr size_t SMEM_BYTES = OFF_AUX + sizeof(Aux);

// Output staging at the CTA's last item, in the K ring: per softmax warp 32 rows
// of 32 floats, padded so that the lanes' 16-byte writes fall in distinct banks.
constexpr int STG_STRIDE = 36;
static_assert((NSM / 32) * 32 * STG_STRIDE * 4 <= KSTAGES * TILEB, "output staging exceeds the K ring");

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

// {2^lo, 2^hi} as two fp16 in one 32-bit word (lo in the low half): the exponents
// are rounded to fp16 first, then raised two at a time by the hardware's
// approximate base-2 exponential (ex2.approx.f16x2; 2^-inf = +0).
__device__ __forceinline__ uint32_t ex2_h2(float lo, float hi) {
    uint32_t x, y;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(x) : "f"(hi), "f"(lo));
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// s0 += lo, s1 += hi for the two fp16 of p (exact products with 1, fp32 sums).
__device__ __forceinline__ void sum_h2(uint32_t p, float &s0, float &s1) {
    asm("{\n\t.reg .b16 a, b, one;\n\t"
        "mov.b32 {a, b}, %2;\n\tmov.b16 one, 0x3C00;\n\t"
        "fma.rn.f32.f16 %0, a, one, %0;\n\tfma.rn.f32.f16 %1, b, one, %1;\n\t}"
        : "+f"(s0), "+f"(s1) : "r"(p));
}

// Packed fp32 pairs (one 64-bit register) for the two-wide FMA.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// True while no wait has given up, agreed by all 32 lanes of the warp (so a
// failure never splits a warp in front of a warp-collective instruction).
__device__ __forceinline__ bool warp_ok(volatile int32_t *fail) { return __all_sync(0xffffffffu, *fail == 0); }

struct ItemInfo {
    int32_t block, t0, t1, pairs;
};

__device__ __forceinline__ ItemInfo item_info(const kvk::PrefillArgs &a, int32_t wi) {
    const kvk::WorkItem w = a.p.work[a.p.cap_dec + wi];
    ItemInfo r;
    r.block = w.block;
    r.t0 = w.t0;
    r.t1 = w.t1;
    r.pairs = (w.t1 - w.t0 + 1) / 2;
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
    const uint32_t sbase = kvd::smem_u32(smem);

    // Launched as a programmatic dependent: library state is read before waiting
    // for the previous kernel only when it was complete before that kernel began;
    // Q, the K/V cache and the outputs are touched only after the wait.
    if (!a.early_ok) kvd::pdl_wait();
    if (tid == 0) kvd::pdl_trigger();   // the split-K merge may be scheduled
    const int32_t *c0 = a.p.cta_item0 + a.gx_dec + 1;
    const int32_t i0 = c0[blockIdx.x];
    const int32_t i1 = c0[blockIdx.x + 1];
    if ((sbase & 1023u) != 0) {
        if (tid == 0) kvd::report(a.err, kvd::DERR_BOUNDS);
        return;
    }
    if (tid == 0) {
        kvd::prefetch_tmap(&tm_k);
        kvd::prefetch_tmap(&tm_v);
        for (int s = 0; s < KSTAGES; ++s) {
            kvd::mbar_init(&x.k_full[s], 1);
            kvd::mbar_init(&x.k_empty[s], 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
            kvd::mbar_init(&x.v_full[s], 1);
            kvd::mbar_init(&x.v_empty[s], 1);
        }
        for (int s = 0; s < MSLOTS; ++s) kvd::mbar_init(&x.meta_full[s], 32);
        kvd::mbar_init(&x.s_full[0], 1);
        kvd::mbar_init(&x.s_full[1], 1);
        kvd::mbar_init(&x.p_full[0], NSM);
        kvd::mbar_init(&x.p_full[1], NSM);
        kvd::mbar_init(&x.pv_done[0], 1);
        kvd::mbar_init(&x.pv_done[1], 1);
        kvd::mbar_init(&x.q_full, NSM);
        kvd::mbar_init(&x.spare, 1);
        kvd::mbar_init(&x.lbar, NSM);
        for (int q = 0; q < 4; ++q) kvd::mbar_init(&x.pbar[q], 128);
        x.fail = 0;
        kvd::fence_mbar_init();
    }
    if (warp == W_MMA) {
        tc::alloc(&x.tmem_base, TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = x.tmem_base;

    if (warp == W_K) {
        // ===================== K producer (whole warp) =====================
        // K of pair g + KSTAGES loads as soon as S of pair g has read K of g.  Each
        // pair's list entries, flags and per-cell visibility are fetched while the K
        // slot is still busy and published through meta_full before the K copy is
        // issued.  V has its own warp: these dependent global reads never hold up a
        // V copy.
        const int32_t lane = tid & 31;
        // (no pass over the items first: the first K copy waits on as few dependent
        // global reads as possible -- work item, tile list, flags)
        int32_t kc = 0;
        int32_t kwi = i0, kj = 0;              // K cursor: item and pair within it
        ItemInfo kit{};
        int32_t kit_wi = -1;                   // the item kit describes
        kvi::DevBlock kb{};
        bool have_k = false;
        int32_t tt[2] = {-1, -1};
        bool full = false;
        bool mhas[4] = {false, false, false, false}, many[4] = {false, false, false, false};
        int32_t mpos[4] = {0, 0, 0, 0};
        long long t_last = clock64();
        // The first pair's K goes out as soon as the previous kernel has finished, from
        // the planner's per-column record (one read, done before the wait); its
        // metadata follows through the loop below, which skips that one copy.
        bool first_out = false;
        {
            const int4 ff = *reinterpret_cast<const int4 *>(a.p.pf_first + 4 * blockIdx.x);
            if (ff.x >= 0) {
                if (lane < 8) {   // warm L2 with the pair's K and V (a prefetch returns nothing)
                    const CUtensorMap *tm = lane < 4 ? &tm_k : &tm_v;
                    const int32_t y = (lane >> 1) & 1 ? ff.y : ff.x;
                    if (y >= 0) kvd::tma_prefetch_2d(tm, hk * 128 + 64 * (lane & 1), y);
                }
                kvd::pdl_wait();   // the K/V cache rows of this ubatch are written
                if (lane == 0) {
                    uint8_t *ks = smem + OFF_K;
                    const int32_t xk = hk * 128;
                    kvd::fence_proxy_async_smem();
                    kvd::mbar_arrive_expect_tx(&x.k_full[0], TILEB);
                    kvd::tma_load_2d(ks, &tm_k, xk, ff.x, &x.k_full[0]);
                    kvd::tma_load_2d(ks + HALF, &tm_k, xk + 64, ff.x, &x.k_full[0]);
                    kvd::tma_load_2d(ks + BOX, &tm_k, xk, ff.y, &x.k_full[0]);
                    kvd::tma_load_2d(ks + HALF + BOX, &tm_k, xk + 64, ff.y, &x.k_full[0]);
                }
                first_out = true;
            }
        }
        while (true) {
            if (!warp_ok(fail)) break;
            bool prog = false;
            {
                if (!have_k) {
                    // the next K load's global reads, done before its slot is free
                    while (kwi < i1) {
                        if (kit_wi != kwi) {
                            kit = item_info(a, kwi);
                            kit_wi = kwi;
                        }
                        if (kj < kit.pairs) break;
                        ++kwi;
                        kj = 0;
                    }
                    if (kwi >= i1) break;      // every pair of every item is loaded
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
                            // some row of the block (positions pos_min .. pos_max) may see it
                            many[r] = has && (!a.u.causal || cp <= kb.pos_max) &&
                                      (a.u.n_swa <= 0 || (int64_t)kb.pos_min - cp < a.u.n_swa);
                        }
                    }
                    have_k = true;
                }
                const int32_t st = kc % KSTAGES;
                bool ready = kc < KSTAGES ||
                             kvd::mbar_test_wait(&x.k_empty[st], (uint32_t)((kc / KSTAGES) - 1) & 1u);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready) {
                    Meta &mt = x.meta[kc % MSLOTS];
                    if (lane == 0) {
                        for (int h = 0; h < 2; ++h)   // a missing second tile: out of bounds, TMA writes zeros
                            mt.ys[h] = tt[h] >= 0 ? kb.stream * a.u.kv_size + tt[h] * TILE : -TILE;
                        mt.full = full ? 1 : 0;
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
                    // the metadata goes out before the K copy is issued
                    kvd::mbar_arrive(&x.meta_full[kc % MSLOTS]);
                    if (kc == 0 && !first_out) {
                        // Warm L2 with the first pair's K and V while the previous kernel
                        // (normally the store of this ubatch's rows) finishes: a prefetch
                        // returns nothing, so racing that kernel's writes is harmless.
                        if (lane < 8) {
                            const CUtensorMap *tm = lane < 4 ? &tm_k : &tm_v;
                            const int32_t y = mt.ys[(lane >> 1) & 1];
                            if (y >= 0) kvd::tma_prefetch_2d(tm, hk * 128 + 64 * (lane & 1), y);
                        }
                        kvd::pdl_wait();   // the K/V cache rows of this ubatch are written
                    }
                    if (lane == 0 && !(kc == 0 && first_out)) {
                        uint8_t *ks = smem + OFF_K + st * TILEB;
                        const int32_t xk = hk * 128;
                        const int32_t y0 = mt.ys[0], y1 = mt.ys[1];
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive_expect_tx(&x.k_full[st], TILEB);
                        kvd::tma_load_2d(ks, &tm_k, xk, y0, &x.k_full[st]);
                        kvd::tma_load_2d(ks + HALF, &tm_k, xk + 64, y0, &x.k_full[st]);
                        kvd::tma_load_2d(ks + BOX, &tm_k, xk, y1, &x.k_full[st]);
                        kvd::tma_load_2d(ks + HALF + BOX, &tm_k, xk + 64, y1, &x.k_full[st]);
                    }
                    ++kc;
                    ++kj;
                    have_k = false;
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
            for (int32_t q = kc > KSTAGES ? kc - KSTAGES : 0; q < kc; ++q)
                (void)kvd::mbar_wait_bounded(&x.k_full[q % KSTAGES], (uint32_t)(q / KSTAGES) & 1u);
        }
    } else if (warp == W_V) {
        // ===================== V producer (whole warp) =====================
        // V of pair g + 3 loads as soon as PV of g is done; the tile coordinates come
        // from the pair's metadata, published by the K producer before its K copy.
        const int32_t lane = tid & 31;
        int32_t total = 0;
        for (int32_t wi = i0; wi < i1; ++wi) total += item_info(a, wi).pairs;
        int32_t vc = 0;
        for (; vc < total; ++vc) {
            const int32_t st = vc % VSTAGES;
            bool ok = __all_sync(0xffffffffu, wait_or_fail(&x.meta_full[vc % MSLOTS], (uint32_t)(vc / MSLOTS) & 1u, fail));
            if (ok && vc >= VSTAGES)
                ok = __all_sync(0xffffffffu,
                                wait_or_fail(&x.v_empty[st], (uint32_t)((vc / VSTAGES) - 1) & 1u, fail));
            if (!ok) break;
            if (vc == 0) kvd::pdl_wait();   // the K/V cache rows of this ubatch are written
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
        }
        if (*fail && lane == 0) {
            for (int32_t q = vc > VSTAGES ? vc - VSTAGES : 0; q < vc; ++q)
                (void)kvd::mbar_wait_bounded(&x.v_full[q % VSTAGES], (uint32_t)(q / VSTAGES) & 1u);
        }
    } else if (warp == W_MMA) {
        // ===================== MMA issuer =====================
        // The tensor core's work per item is a fixed sequence: S_0, S_1, then for
        // each pair j: PV_j, S_j+2 (S_j+2 goes to the score buffer of pair j, whose P
        // PV_j reads first: one thread's MMAs run in issue order).  Every step waits
        // on its mbarrier with a blocking (suspending, bounded) wait, so the thread
        // wakes as soon as a P or a K tile is ready.
        if ((tid & 31) == 0) {
            int32_t gidx = 0;                  // global pair-tile counter (stage rings)
            uint32_t n_q = 0;
            bool ok = true;
            auto issue_s = [&](int32_t gi, int32_t buf) -> bool {
                if (!wait_or_fail(&x.k_full[gi % KSTAGES], (uint32_t)(gi / KSTAGES) & 1u, fail)) return false;
                tc::fence_after();
                const uint32_t k_addr = sbase + OFF_K + (gi % KSTAGES) * TILEB;
                const uint32_t d = tmem + (uint32_t)buf * 128u;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF + (uint32_t)(kk & 3) * 32u;
                    tc::mma_ts(d, tmem + COL_Q + 8u * (uint32_t)kk, tc::sdesc_sw128(k_addr + off, 16, 1024),
                               IDESC_S, kk > 0 ? 1u : 0u);
                }
                tc::commit(&x.s_full[buf]);
                tc::commit(&x.k_empty[gi % KSTAGES]);   // this K tile is consumed
                return true;
            };
            for (int32_t wi = i0; wi < i1 && ok; ++wi) {
                const ItemInfo it = item_info(a, wi);
                if (it.pairs == 0) continue;
                if (!(ok = wait_or_fail(&x.q_full, n_q & 1u, fail))) break;
                ++n_q;
                tc::fence_after();
                ok = issue_s(gidx, 0);
                if (ok && it.pairs > 1) ok = issue_s(gidx + 1, 1);
                for (int32_t j = 0; j < it.pairs && ok; ++j) {
                    // P of pair gp is signalled on p_full[gp & 1]
                    const int32_t gp = gidx + j;
                    if (!(ok = wait_or_fail(&x.p_full[gp & 1], (uint32_t)(gp >> 1) & 1u, fail))) break;
                    if (!(ok = wait_or_fail(&x.v_full[gp % VSTAGES], (uint32_t)(gp / VSTAGES) & 1u, fail))) break;
                    tc::fence_after();
                    const uint32_t v_addr = sbase + OFF_V + (gp % VSTAGES) * TILEB;
                    const uint32_t p_tmem = tmem + 128u * (uint32_t)(j & 1);
                    // O += P V over the 128 cells: P of cells 16kk .. 16kk + 15 is 8 TMEM
                    // columns at 32 (kk / 2) + 8 (kk % 2) of the score buffer (each softmax
                    // thread writes its 32 cells' P at the start of its own 32 S columns)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        tc::mma_ts(tmem + COL_O, p_tmem + 32u * (uint32_t)(kk >> 1) + 8u * (uint32_t)(kk & 1),
                                   tc::sdesc_sw128(v_addr + (uint32_t)kk * 2048u, HALF, 1024), IDESC_PV,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(&x.pv_done[gp & 1]);
                    tc::commit(&x.v_empty[gp % VSTAGES]);
                    if (j + 2 < it.pairs) ok = issue_s(gidx + j + 2, j & 1);
                }
                gidx += it.pairs;
            }
            // all issued MMAs complete before TMEM is released
            tc::commit(&x.spare);
            (void)kvd::mbar_wait_bounded(&x.spare, 0);
        }
    } else {
        // ============ softmax / correction / epilogue (warps 0-15, four threads per row) ============
        // Warps w, w + 4, w + 8 and w + 12 share TMEM lane quarter w: thread (n, qd) owns
        // cells 32qd .. 32qd + 31 of every pair tile of row n and d = 32qd .. 32qd + 31
        // of O.  The four threads of a row exchange their maxima once per pair through
        // an mbarrier of their four warps (arrive, then a bounded wait, never bar.sync:
        // if a wait elsewhere gives up, the partners time out instead of hanging).
        const int32_t n = tid & 127;           // TMEM lane = query vector
        const int32_t qd = tid >> 7;           // cell quarter, and d quarter of O
        const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_mine = tmem + lane_q + (uint32_t)(32 * qd);   // + 128 * score buffer
        const uint32_t o_mine = tmem + lane_q + COL_O + (uint32_t)(32 * qd);
        uint64_t *pbar = &x.pbar[warp & 3];
        uint32_t n_s0 = 0, n_s1 = 0;           // score-buffer phases (scalars: no local memory)
        uint32_t n_l = 0, n_p = 0;
        int32_t k = 0;                         // pair tiles consumed (stage ring position)
        bool ok = true;
        bool dep_done = false;                 // waited for the previous kernel of the stream
        for (int32_t wi = i0; wi < i1 && ok && warp_ok(fail); ++wi) {
            const ItemInfo it = item_info(a, wi);
            const int32_t nitems = a.p.blk_nitems[it.block];   // used at the item's end
            // the query vector behind my TMEM lane (an empty item has a block that sees
            // no cell: zeros, or an empty partial), fetched here rather than from the
            // producer so that Q starts loading as early as possible
            int32_t row = -1, rpos = 0;
            if (wi == i0) {
                row = a.p.pf_rows[blockIdx.x * M + n];   // written by the planner
            } else {
                const kvi::DevBlock b = a.u.blocks[it.block];
                if (n < b.n_rows * G) row = a.u.perm[b.row0 + n / G];
            }
            if (row >= 0) rpos = a.u.rows[row].pos;
            const bool live = row >= 0;
            const int32_t h = hk * G + (n % G);
            if (!dep_done) {   // before the first read of Q and the first write of an output
                // warm L2 with my 64 bytes of Q while the previous kernel finishes (a
                // prefetch returns nothing, so racing its writes is harmless)
                if (live && it.pairs > 0) kvd::prefetch_l2(a.q + ((int64_t)row * a.n_head + h) * 128 + 32 * qd);
                kvd::pdl_wait();
                dep_done = true;
            }
            float m_run = -INFINITY, l_run = 0.f;   // the row's running maximum, this quarter's row sum
            if (it.pairs > 0) {
            // ---- Q into TMEM (the A operand of S = Q K^T): row n, d quarter qd, fp16,
            //      two values per 32-bit column ----
            {
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(a.q + ((int64_t)(live ? row : 0) * a.n_head + h) * 128 + 32 * qd);
                uint32_t qw[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = live ? src[c] : make_uint4(0, 0, 0, 0);
                    qw[4 * c + 0] = v.x;
                    qw[4 * c + 1] = v.y;
                    qw[4 * c + 2] = v.z;
                    qw[4 * c + 3] = v.w;
                }
                tc::st16(tmem + lane_q + COL_Q + 16u * (uint32_t)qd, qw);
                tc::wait_st();
                tc::fence_before();
                kvd::mbar_arrive(&x.q_full);
            }
            for (int32_t j = 0; j < it.pairs; ++j, ++k) {
                const int32_t st = k % VSTAGES;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.meta_full[k % MSLOTS], (uint32_t)(k / MSLOTS) & 1u, fail));
                if (!ok) break;
                const Meta &mt = x.meta[k % MSLOTS];
                const bool full = mt.full != 0;
                const uint32_t ns = (j & 1) ? n_s1 : n_s0;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.s_full[j & 1], ns & 1u, fail));
                if (!ok) break;
                if (j & 1) ++n_s1; else ++n_s0;
                tc::fence_after();
                // ---- my 32 columns of S -> registers (one TMEM read, warp collective);
                //      masked -> -inf ----
                const uint32_t s_addr = s_mine + (uint32_t)(j & 1) * 128u;
                uint32_t sb[32];
                tc::ld32(s_addr, sb);
                if (!live) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) sb[c] = __float_as_uint(-INFINITY);
                } else if (!full) {
                    // which of my 32 cells this row sees (16-byte loads, all issued before
                    // any test), applied as a 32-bit mask
                    uint4 hb[2];
                    int4 cp[8];
                    const uint4 *hs = reinterpret_cast<const uint4 *>(&mt.has[32 * qd]);
                    const int4 *cs = reinterpret_cast<const int4 *>(&mt.cpos[32 * qd]);
#pragma unroll
                    for (int q = 0; q < 2; ++q) hb[q] = hs[q];
#pragma unroll
                    for (int q = 0; q < 8; ++q) cp[q] = cs[q];
                    // the positions this row sees (causal order, sliding window)
                    const kvd::PosRange rr = kvd::pos_range(a.u.causal, a.u.n_swa, rpos);
                    uint32_t vm = 0;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t hw = (&hb[q >> 2].x)[q & 3];   // has of cells 4q .. 4q + 3
                        const int32_t c4[4] = {cp[q].x, cp[q].y, cp[q].z, cp[q].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool vis = ((hw >> (8 * e)) & 0xffu) != 0 && kvd::pos_in(rr, c4[e]);
                            vm |= (uint32_t)vis << (4 * q + e);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        sb[c] = ((vm >> c) & 1u) ? sb[c] : __float_as_uint(-INFINITY);
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(sb[c]), __uint_as_float(sb[c + 1]));
                // ---- the row maximum over the four quarters (partners: the same lane of
                //      warps w, w + 4, w + 8, w + 12) ----
                x.red[j & 1][qd][n] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                kvd::mbar_arrive(pbar);
                ok = __all_sync(0xffffffffu, wait_or_fail(pbar, n_p & 1u, fail));
                ++n_p;
                if (!ok) break;
                const float tmax = fmaxf(fmaxf(x.red[j & 1][0][n], x.red[j & 1][1][n]),
                                         fmaxf(x.red[j & 1][2][n], x.red[j & 1][3][n])) * a.scale_log2;
                const float m_new = fmaxf(m_run, tmax);
                const bool grow = m_new > m_run + RESCALE_LOG2 || (m_run == -INFINITY && m_new != -INFINITY);
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2_approx(m_run - m_new);
                    m_run = m_new;
                    l_run *= alpha;
                }
                // ---- P = 2^(s*scale - m) as fp16 at the start of my S columns: my 32 cells
                //      are 16 columns (two fp16 per column, lower cell in the low half);
                //      the exponent s*scale - m is rounded to fp16 and two of them are
                //      raised at once (ex2.approx.f16x2), which yields P in the fp16 the PV
                //      product reads; the row sum adds those same fp16 values in fp32 ----
                {
                    // no maximum yet (nothing visible so far, or a lane past the block):
                    // subtract +inf so that every exponent is -inf and P is 0
                    const float nm = m_run != -INFINITY ? -m_run : -INFINITY;
                    const uint64_t sc2 = pk2(a.scale_log2, a.scale_log2), nm2 = pk2(nm, nm);
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
                    uint32_t pw[16];
#pragma unroll
                    for (int c2 = 0; c2 < 16; ++c2) {
                        const int c = 2 * c2;
                        float x0, x1;
                        upk2(ffma2(pk2(__uint_as_float(sb[c]), __uint_as_float(sb[c + 1])), sc2, nm2), x0, x1);
                        const uint32_t p2 = ex2_h2(x0, x1);
                        pw[c2] = p2;
                        sum_h2(p2, ls[(c2 & 1) * 2], ls[(c2 & 1) * 2 + 1]);
                    }
                    l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    tc::st16(s_addr, pw);
                }
                // ---- O *= alpha where the row's running maximum moved (rare), my 32
                //      columns; O is stable once PV of pair k - 1 finished ----
                if (j > 0 && __any_sync(0xffffffffu, grow)) {
                    ok = __all_sync(0xffffffffu,
                                    wait_or_fail(&x.pv_done[(k - 1) & 1], (uint32_t)((k - 1) >> 1) & 1u, fail));
                    if (!ok) break;
                    tc::fence_after();
                    uint32_t r[32];
                    tc::ld32(o_mine, r);
#pragma unroll
                    for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                    tc::st32(o_mine, r);
                }
                if (!full && qd < 2) {
                    // V rows of cells nobody in the block sees: zero (P is 0 there; V may
                    // be garbage); thread (n, qd < 2) clears d half qd of cell n
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.v_full[st], (uint32_t)(k / VSTAGES) & 1u, fail));
                    if (!ok) break;
                    if (!mt.anyvis[n]) {
                        uint8_t *vs = smem + OFF_V + st * TILEB + qd * HALF + n * 128;
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
            // ---- wait for the item's last PV (pair k - 1) ----
            ok = __all_sync(0xffffffffu,
                            wait_or_fail(&x.pv_done[(k - 1) & 1], (uint32_t)((k - 1) >> 1) & 1u, fail));
            if (!ok) break;
            tc::fence_after();
            }   // it.pairs > 0
            // ---- the row sum over the four quarters (double-buffered by item parity) ----
            x.lex[n_l & 1][qd][n] = l_run;
            kvd::mbar_arrive(&x.lbar);
            ok = __all_sync(0xffffffffu, wait_or_fail(&x.lbar, n_l & 1u, fail));
            if (!ok) break;
            const float l_tot = (x.lex[n_l & 1][0][n] + x.lex[n_l & 1][1][n]) +
                                (x.lex[n_l & 1][2][n] + x.lex[n_l & 1][3][n]);
            ++n_l;
            float *dst = nullptr;
            float sc = 1.f;
            if (nitems == 1) {
                if (live) dst = a.o + ((int64_t)row * a.n_head + h) * 128 + 32 * qd;
                sc = l_tot > 0.f ? 1.f / l_tot : 0.f;
            } else {
                // a split block: this item's partial (its slot is its index among the
                // prefill items); k_merge_pf combines the partials after the kernel
                float *pp = a.part + (((int64_t)wi * a.n_head_kv + hk) * M + n) * PART_STRIDE;
                if (qd == 0) {
                    pp[0] = m_run;
                    pp[1] = l_tot;
                }
                dst = pp + 4 + 32 * qd;
            }
            uint32_t r[32];
            if (it.pairs > 0) {                  // item-uniform: the TMEM read stays warp collective
                tc::ld32(o_mine, r);
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) r[c] = 0u;
            }
            if (wi + 1 == i1) {
                // The CTA's last item: the K ring is idle (every S has completed), so each
                // warp stages its 32 rows there and writes them out row by row, 8 lanes
                // per 128-byte row, instead of one row per lane.
                float *stg = reinterpret_cast<float *>(smem + OFF_K) + warp * (32 * STG_STRIDE);
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4 *>(stg + (tid & 31) * STG_STRIDE + c) =
                        make_float4(__uint_as_float(r[c + 0]) * sc, __uint_as_float(r[c + 1]) * sc,
                                    __uint_as_float(r[c + 2]) * sc, __uint_as_float(r[c + 3]) * sc);
                __syncwarp();
                const int32_t lane = tid & 31, part = lane & 7;
#pragma unroll 4
                for (int i = 0; i < 8; ++i) {
                    const int32_t rr = 4 * i + (lane >> 3);   // the warp's row (its lane)
                    float *d = reinterpret_cast<float *>(
                        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), rr));
                    if (d)
                        *reinterpret_cast<float4 *>(d + 4 * part) =
                            *reinterpret_cast<const float4 *>(stg + rr * STG_STRIDE + 4 * part);
                }
            } else if (dst) {
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    float4 v;
                    v.x = __uint_as_float(r[c + 0]) * sc;
                    v.y = __uint_as_float(r[c + 1]) * sc;
                    v.z = __uint_as_float(r[c + 2]) * sc;
                    v.w = __uint_as_float(r[c + 3]) * sc;
                    *reinterpret_cast<float4 *>(dst + c) = v;
                }
            }
            tc::fence_before();
        }
    }

    tc::fence_before();
    __syncthreads();
    if (*fail && tid == 0) kvd::report(a.err, kvd::DERR_MMA_TIMEOUT);
    if (warp == W_MMA) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }

}


// Split-K merge of the prefill path: sixteen 128-thread CTAs per (prefill block,
// KV head), 8 query vectors each; blocks covered by a single item were written
// directly and return at once.  Thread t takes query vector 8z + t / 16 and 8 of
// its 128 values, and loads up to four partials at once, folding them into a
// running (M, L, O):
//   O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q.
// Launched as a programmatic dependent of the attention kernel: the plan is
// read first, the partials only after the attention grid has finished.  The
// CTAs are small (128 threads, at most 64 registers each); they take the SMs as
// the attention CTAs retire (capping them at 48 registers, so that one would
// wait beside each attention CTA, measured slower: two partials per round trip).
constexpr int MERGE_SPLIT = 16;
constexpr int MERGE_QMAX = 4;

__global__ void __launch_bounds__(128, 8) k_merge_pf(const kvk::PrefillArgs a) {
    const int32_t b = a.u.n_dec_blocks + blockIdx.x;
    const int32_t hk = blockIdx.y;
    const int32_t nitems = a.p.blk_nitems[b];
    if (nitems <= 1) {
        kvd::pdl_trigger();
        return;
    }
    const kvi::DevBlock blk = a.u.blocks[b];
    const int32_t n = (int32_t)blockIdx.z * (M / MERGE_SPLIT) + (int32_t)(threadIdx.x >> 4);   // 8 per CTA
    const int32_t d0 = (int32_t)(threadIdx.x & 15) * 8;
    const int32_t G = a.gqa;
    if (n >= blk.n_rows * G) return;
    const int32_t row = a.u.perm[blk.row0 + n / G];
    const int32_t h = hk * G + (n % G);
    const int32_t first = a.p.blk_item0[b] - a.p.cap_dec;
    const int64_t istride = (int64_t)a.n_head_kv * M * PART_STRIDE;
    const float *pr = a.part + (((int64_t)first * a.n_head_kv + hk) * M + n) * PART_STRIDE;
    kvd::pdl_wait();
    kvd::pdl_trigger();   // the next kernel (a K/V store) may be scheduled
    float mx = -INFINITY, L = 0.f;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    for (int32_t q0 = 0; q0 < nitems; q0 += MERGE_QMAX) {
        float mk[MERGE_QMAX], lk[MERGE_QMAX];
        float4 v0[MERGE_QMAX], v1[MERGE_QMAX];
#pragma unroll
        for (int i = 0; i < MERGE_QMAX; ++i) {
            mk[i] = -INFINITY;
            lk[i] = 0.f;
            v0[i] = v1[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q0 + i < nitems) {
                const float *pq = pr + (int64_t)(q0 + i) * istride;
                mk[i] = __ldcg(pq);
                lk[i] = __ldcg(pq + 1);
                v0[i] = __ldcg(reinterpret_cast<const float4 *>(pq + 4 + d0));
                v1[i] = __ldcg(reinterpret_cast<const float4 *>(pq + 4 + d0) + 1);
            }
        }
        float mr = -INFINITY;
#pragma unroll
        for (int i = 0; i < MERGE_QMAX; ++i) mr = fmaxf(mr, mk[i]);
        const float mn = fmaxf(mx, mr);
        if (mn == -INFINITY) continue;
        const float al = mx == -INFINITY ? 0.f : ex2_approx(mx - mn);
        L *= al;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] *= al;
#pragma unroll
        for (int i = 0; i < MERGE_QMAX; ++i) {
            const float sc = mk[i] == -INFINITY ? 0.f : ex2_approx(mk[i] - mn);
            L = fmaf(lk[i], sc, L);
            acc[0] = fmaf(v0[i].x, sc, acc[0]);
            acc[1] = fmaf(v0[i].y, sc, acc[1]);
            acc[2] = fmaf(v0[i].z, sc, acc[2]);
            acc[3] = fmaf(v0[i].w, sc, acc[3]);
            acc[4] = fmaf(v1[i].x, sc, acc[4]);
            acc[5] = fmaf(v1[i].y, sc, acc[5]);
            acc[6] = fmaf(v1[i].z, sc, acc[6]);
            acc[7] = fmaf(v1[i].w, sc, acc[7]);
        }
        mx = mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float4 *dst = reinterpret_cast<float4 *>(a.o + ((int64_t)row * a.n_head + h) * 128 + d0);
    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
}

}  // namespace

namespace kvk {

cudaError_t load_prefill_kernels() {
    cudaError_t e = cudaFuncSetAttribute(k_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, k_merge_pf);
}

// The shared-memory attribute was set for the current device by load_prefill_kernels.
cudaError_t launch_prefill(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const PrefillArgs &a,
                           int32_t grid_x, cudaStream_t st) {
    // Both kernels are programmatic dependents of the kernel before them: the
    // attention kernel sets up (and, with early_ok, reads its plan) while the K/V
    // store finishes; the merge reads the plan while the attention kernel runs.
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, a.n_head_kv);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_prefill, *tm_k, *tm_v, a);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(a.u.n_blocks - a.u.n_dec_blocks, a.n_head_kv, MERGE_SPLIT);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, k_merge_pf, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kvk
