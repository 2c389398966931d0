// K3b: GQA flash attention, prefill / mixed path, on tcgen05 tensor cores.
//
// "llama.cpp and the ubatch", "Chunked prefill is the same mechanism": a
// chunk of U rows against C cached cells is a [U, C+U] score matrix; with the
// mask of "The mask is doing the work" (occupied, same first sequence id,
// not later) it is the same softmax(q K^T / sqrt(d) + mask) V as decode, but
// now a dense contraction worth putting on the tensor cores.
//
// Design (sm_103a, one CTA of 384 threads per SM):
//  * a block = up to 256 query vectors (rows sharing a stream and first
//    sequence id, times the GQA group), held as two 128-lane MMA tiles A
//    (query vectors 0..127) and B (128..255) that share every K/V tile; a work
//    item = one block, one KV head, a chunk of the block's list of visible
//    64-cell tiles, consumed two at a time (one step = 128 cells);
//  * TMEM (512 columns): S_A, S_B (fp32 scores, 128 columns each; P is written
//    over the first 64 as fp16 pairs), O_A, O_B (fp32, d = 0..127);
//  * shared memory: Q_A, Q_B (written by the softmax threads, 128-byte
//    swizzle), a 2-stage K ring and a 2-stage V ring of 128-cell tiles (TMA,
//    128-byte swizzle), a ring of per-step metadata;
//  * warp 8 streams K tiles and the steps' metadata (list entries, flags, the
//    cells' positions and sequence membership), warp 10 streams V tiles, one
//    thread of warp 9 issues the MMAs in the order
//        S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
//    so that the tensor core works on one tile while the other tile's softmax
//    runs (S = Q K^T as SS-MMA M128 N128 K16 x 8; O += P V as TS-MMA with P
//    read from TMEM);
//  * warps 0-3 (tile A) and 4-7 (tile B): one thread per query vector (TMEM
//    lane) holds the row's 128 scores of a step, applies the per-cell mask on
//    steps that are not fully visible, takes the row maximum locally, runs the
//    online softmax in base 2 (exponents rounded to fp16, two per
//    ex2.approx.f16x2), writes P and rescales its O row only when the running
//    maximum grew by more than 2^8 (otherwise the stale maximum is kept; the
//    final normalisation uses the same one);
//  * cells nobody in the block may see get their V rows zeroed in shared
//    memory before the PV product (P is 0 there, but 0 * NaN would not be);
//  * a block split over several CTAs leaves one partial (m, l, O) per piece;
//    the CTAs whose last item is a piece of that block wait (bounded) until
//    every piece is counted and merge a share of its query vectors each, so no
//    second kernel is needed.  (Only a column's last item waits, and a split
//    block's other pieces are either the last item of an earlier column or the
//    first of a later one, so every wait ends.)  Every wait is bounded.

#include "dev_common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace {

using kvi::TILE;
using kvi::PF_M;

constexpr int NT = 384;                  // 12 warps
constexpr int W_K = 8;                   // K producer + metadata
constexpr int W_MMA = 9;                 // TMEM allocation and MMA issue
constexpr int W_V = 10;                  // V producer
constexpr int W_Q = 11;                  // Q producer (TMA), when the launch loads Q that way
constexpr int NSM = 256;                 // softmax threads (warps 0-7)
constexpr int M = 128;                   // lanes of one MMA tile
static_assert(PF_M == 2 * M, "a prefill block is two MMA tiles");
constexpr int HALF = 128 * 128;          // [128 rows][64 fp16], 128-byte rows
constexpr int TILEB = 2 * HALF;          // 32 KiB: 128 rows x 128 fp16
constexpr int BOX = 64 * 128;            // one TMA box: 64 rows x 64 fp16
constexpr int KSTAGES = 2;
constexpr int VSTAGES = 2;
constexpr int OFF_Q = 0;                 // Q_A, Q_B
constexpr int OFF_K = 2 * TILEB;
constexpr int OFF_V = OFF_K + KSTAGES * TILEB;
constexpr int OFF_AUX = OFF_V + VSTAGES * TILEB;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0;            // + 128 * tile
constexpr uint32_t COL_O = 256;          // + 128 * tile
constexpr float RESCALE_LOG2 = 8.0f;
// Register split (setmaxnreg, per warpgroup): the kernel is launched with
// LAUNCH_REGS registers per thread (the build checks ptxas's count); the two
// softmax warpgroups take SM_REGS each, the producer / MMA warpgroup gives back
// down to PR_REGS.  The shares must not exceed what the launch holds, or the
// increase would wait forever.
constexpr int LAUNCH_REGS = 168;
constexpr int SM_REGS = 224;
constexpr int PR_REGS = 56;
static_assert(LAUNCH_REGS * NT <= 65536, "launch registers");
static_assert(2 * 128 * SM_REGS + 128 * PR_REGS <= LAUNCH_REGS * NT, "register split exceeds the launch's registers");
static_assert(SM_REGS % 8 == 0 && PR_REGS % 8 == 0 && PR_REGS >= 24 && SM_REGS <= 256, "setmaxnreg counts");
constexpr unsigned POLL_NS = 32;

constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16(128, 128, 0, 1);

// Metadata ring.  The slot of step g is rewritten for step g + MSLOTS once the
// K stage of step g + MSLOTS - KSTAGES is free, i.e. after S_A and S_B of that
// step completed; those were issued after PV_A and PV_B of the step before,
// which waited for both tiles' softmax of that step -- so both softmax groups
// are past step g + MSLOTS - KSTAGES - 1 >= g + 1, and the V producer, which
// issued V of that step, is past g too.
constexpr int MSLOTS = 6;
static_assert(MSLOTS >= KSTAGES + 2, "metadata ring too short for the K ring");

struct __align__(16) Meta {     // per step: what the K producer learned about its 128 cells
    int32_t full;             // every row of the block sees every cell
    int32_t ys[2];            // TMA row coordinates of the two 64-cell halves
    int32_t pad;
    int32_t cpos[128];
    uint32_t has[4];          // bit c: cell 32 r + c holds the block's sequence, not from a later ubatch
    uint32_t anyvis[4];       // ... and some row of the block may see it
};

struct __align__(16) Aux {
    uint64_t k_full[KSTAGES], k_empty[KSTAGES], v_full[VSTAGES], v_empty[VSTAGES];
    uint64_t meta_full[MSLOTS];
    uint64_t s_full[2], p_full[2], pv_done[2], q_full[2];   // [tile]
    uint64_t qt_full[2];      // [tile] Q landed by TMA (1 arrival + bytes)
    uint64_t q_free[2];       // [tile] the item's epilogue is done with the Q area (128 arrivals)
    uint64_t wbar;            // the softmax threads meet (256 arrivals)
    uint64_t gbar;            // a merge may start: every piece of the block is counted (1 arrival)
    uint64_t mbar;            // the partials of one merge pass are in shared memory (bulk copies)
    uint64_t spare;
    uint32_t tmem_base;
    int32_t fail;
    int32_t mrg_lo, mrg_hi;   // this CTA's share of the merged block's query vectors
    Meta meta[MSLOTS];
    float2 mlx[PF_M];         // with clusters: this CTA's piece's (m, l) per query vector
};

constexpr size_t SMEM_BYTES = OFF_AUX + sizeof(Aux);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

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

// True while no wait has given up, agreed by all 32 lanes of the warp (so a
// failure never splits a warp in front of a warp-collective instruction).
__device__ __forceinline__ bool warp_ok(volatile int32_t *fail) { return __all_sync(0xffffffffu, *fail == 0); }

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

// 1/x with the hardware's approximate reciprocal (rcp.approx.ftz: about 1 ulp).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ int32_t ld_acquire(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// S = Q K^T of one tile: 8 SS-MMAs (K = 16 each) over d = 0..127; a0 / b0 are the
// descriptors of Q and of the K stage, advanced by the 32-byte K steps inside a
// 128-byte swizzled row and by the second d half.  The bases go through an opaque
// move first, so that the eight offset descriptors are formed next to their MMA
// (one add each) instead of all being kept in registers across the issue loop;
// forming a whole descriptor per MMA would cost the issuing thread more than the
// tensor pipe takes for the MMA.
__device__ __forceinline__ void issue_s8(uint32_t d, uint64_t a0, uint64_t b0) {
    asm volatile("" : "+l"(a0), "+l"(b0));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * HALF + (kk & 3) * 32) >> 4);
        tc::mma_ss(d, a0 + off, b0 + off, IDESC_S, kk > 0 ? 1u : 0u);
    }
}

// O += P V of one tile: 8 TS-MMAs (16 cells each); P of cells 16kk .. 16kk + 15 is
// 8 TMEM columns at p + 8kk, V (MN-major) rows 16kk .. at b0 + 2 KiB kk.
__device__ __forceinline__ void issue_pv8(uint32_t d, uint32_t p, uint64_t b0, uint32_t acc) {
    asm volatile("" : "+l"(b0), "+r"(p));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        tc::mma_ts(d, p + 8u * (uint32_t)kk, b0 + (uint64_t)((kk * 2048) >> 4), IDESC_PV, (acc | (uint32_t)kk) ? 1u : 0u);
}

struct ItemInfo {
    int32_t block, t0, t1, steps;
};

__device__ __forceinline__ ItemInfo item_info(const kvk::PrefillArgs &a, int32_t wi) {
    const kvk::WorkItem w = a.p.work[a.p.cap_dec + wi];
    ItemInfo r;
    r.block = w.block;
    r.t0 = w.t0;
    r.t1 = w.t1;
    r.steps = (w.t1 - w.t0 + 1) / 2;
    return r;
}

// Is prefill item wi the last item of its CTA column?  (A column's items are
// consecutive.)
__device__ __forceinline__ bool last_of_column(const kvk::PrefillArgs &a, int32_t wi, int32_t n_items) {
    return wi + 1 >= n_items || a.p.work[a.p.cap_dec + wi + 1].cta != a.p.work[a.p.cap_dec + wi].cta;
}

__global__ void __launch_bounds__(NT, 1)
k_prefill(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
          const __grid_constant__ CUtensorMap tm_part, const __grid_constant__ CUtensorMap tm_q,
          const kvk::PrefillArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Aux &x = *reinterpret_cast<Aux *>(smem + OFF_AUX);
    volatile int32_t *fail = &x.fail;
    const int32_t tid = threadIdx.x;
    const int32_t warp = tid >> 5;
    const int32_t lane = tid & 31;
    const int32_t hk = blockIdx.y;
    const int32_t G = a.gqa;
    const uint32_t sbase = kvd::smem_u32(smem);

    // Launched as a programmatic dependent: library state is read before waiting
    // for the previous kernel only when it was complete before that kernel began;
    // Q, the K/V cache, the outputs, the partials and the merge counters are
    // touched only after the wait.
    if (!a.early_ok) kvd::pdl_wait();
    // The next kernel of the stream (normally the next call's K/V store) may be
    // scheduled now: it waits for this grid's completion before it touches memory,
    // and meanwhile its launch and its own start-up overlap this kernel.
    if (tid == 0) kvd::pdl_trigger();
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
        kvd::prefetch_tmap(&tm_part);
        for (int s = 0; s < KSTAGES; ++s) {
            kvd::mbar_init(&x.k_full[s], 1);
            kvd::mbar_init(&x.k_empty[s], 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
            kvd::mbar_init(&x.v_full[s], 1);
            kvd::mbar_init(&x.v_empty[s], 1);
        }
        for (int s = 0; s < MSLOTS; ++s) kvd::mbar_init(&x.meta_full[s], 32);
        for (int t = 0; t < 2; ++t) {
            kvd::mbar_init(&x.s_full[t], 1);
            kvd::mbar_init(&x.p_full[t], M);
            kvd::mbar_init(&x.pv_done[t], 1);
            kvd::mbar_init(&x.q_full[t], M);
            kvd::mbar_init(&x.qt_full[t], 1);
            kvd::mbar_init(&x.q_free[t], M);
        }
        kvd::mbar_init(&x.wbar, NSM);
        kvd::mbar_init(&x.gbar, 1);
        kvd::mbar_init(&x.mbar, 1);
        kvd::mbar_init(&x.spare, 1);
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
    // With clusters: this CTA's last item is a piece of a block split over its cluster
    // (its partial staged in shared memory), merged after the cluster's first barrier.
    bool mrg_cl = false;
    int32_t mrg_nq = 0, mrg_row0 = 0;
    if (warp >= 8) {
    // register split, one instruction per warpgroup: warps 8-11 give registers back
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PR_REGS));
    if (warp == W_K) {
        // ===================== K producer (whole warp) =====================
        // K of step g + KSTAGES loads as soon as S_A and S_B of step g have read K
        // of g.  Each step's list entries, flags and per-cell visibility are
        // fetched while the K slot is still busy and published through meta_full
        // before the K copy is issued.
        int32_t kc = 0;
        int32_t kwi = i0, kj = 0;              // K cursor: item and step within it
        ItemInfo kit{};
        int32_t kit_wi = -1;
        kvi::DevBlock kb{};
        bool have_k = false;
        int32_t tt[2] = {-1, -1};
        bool full = false;
        uint32_t mhas = 0, many = 0;           // bit r: cell lane + 32 r
        int32_t mpos[4] = {0, 0, 0, 0};
        long long t_last = clock64();
        // The first step's K goes out as soon as the previous kernel has finished, from
        // the planner's per-column record (one read, done before the wait); its
        // metadata follows through the loop below, which skips that one copy.
        bool first_out = false;
        {
            const int4 ff = *reinterpret_cast<const int4 *>(a.p.pf_first + 4 * blockIdx.x);
            if (ff.x >= 0) {
                if (lane < 8) {   // warm L2 with the step's K and V (a prefetch returns nothing)
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
            if (!have_k) {
                // the next K load's global reads, done before its slot is free
                while (kwi < i1) {
                    if (kit_wi != kwi) {
                        kit = item_info(a, kwi);
                        kit_wi = kwi;
                    }
                    if (kj < kit.steps) break;
                    ++kwi;
                    kj = 0;
                }
                if (kwi >= i1) break;      // every step of every item is loaded
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
                mhas = many = 0;
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
                        mpos[r] = cp;
                        // some row of the block (positions pos_min .. pos_max) may see it
                        const bool any = has && (!a.u.causal || cp <= kb.pos_max) &&
                                         (a.u.n_swa <= 0 || (int64_t)kb.pos_min - cp < a.u.n_swa);
                        mhas |= (has ? 1u : 0u) << r;
                        many |= (any ? 1u : 0u) << r;
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
                        mt.cpos[lane + 32 * r] = mpos[r];
                        const uint32_t hb = __ballot_sync(0xffffffffu, (mhas >> r) & 1u);
                        const uint32_t ab = __ballot_sync(0xffffffffu, (many >> r) & 1u);
                        if (lane == 0) {
                            mt.has[r] = hb;
                            mt.anyvis[r] = ab;
                        }
                    }
                }
                __syncwarp();
                // the metadata goes out before the K copy is issued
                kvd::mbar_arrive(&x.meta_full[kc % MSLOTS]);
                if (kc == 0 && !first_out) {
                    // Warm L2 with the first step's K and V while the previous kernel
                    // (normally the store of this ubatch's rows) finishes.
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
        // V of step g + VSTAGES loads as soon as PV_A and PV_B of g are done; the
        // tile coordinates come from the step's metadata.
        int32_t total = 0;
        for (int32_t wi = i0; wi < i1; ++wi) total += item_info(a, wi).steps;
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
                const Meta &mt = x.meta[vc % MSLOTS];
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
    } else if (warp == W_Q) {
        // ===================== Q producer (launches with a.q_tma) =====================
        // Per item with a step, per tile with query vectors: once the tile's previous
        // such item is done with the Q area (its epilogue staged output there), Q
        // arrives as two (64, gqa, 128 / gqa) boxes -- query vector n of the tile is
        // row n of the 128-byte-swizzled tile, the A operand layout of S = Q K^T.
        if (a.q_tma && lane == 0) {
            uint32_t nt[2] = {0, 0};           // items loaded per tile
            bool dep = false;
            for (int32_t wi = i0; wi < i1; ++wi) {
                const ItemInfo it = item_info(a, wi);
                if (it.steps == 0) continue;
                const kvi::DevBlock b = a.u.blocks[it.block];
                bool ok = true;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (t == 1 && b.n_rows * G <= M) break;
                    if (nt[t] > 0) ok = wait_or_fail(&x.q_free[t], (nt[t] - 1) & 1u, fail);
                    if (!ok) break;
                    if (!dep) {
                        kvd::pdl_wait();   // Q comes from before the previous kernel of the stream
                        dep = true;
                    }
                    uint8_t *qs = smem + OFF_Q + t * TILEB;
                    const int32_t tok = b.tok0 + (M * t) / G;
                    kvd::mbar_arrive_expect_tx(&x.qt_full[t], TILEB);
                    kvd::tma_load_3d(qs, &tm_q, 0, hk * G, tok, &x.qt_full[t]);
                    kvd::tma_load_3d(qs + HALF, &tm_q, 64, hk * G, tok, &x.qt_full[t]);
                    ++nt[t];
                }
                if (!ok) break;
            }
            // loads already issued land before the CTA exits
            if (*fail)
                for (int t = 0; t < 2; ++t)
                    if (nt[t] > 0) (void)kvd::mbar_wait_bounded(&x.qt_full[t], (nt[t] - 1) & 1u);
        }
    } else if (warp == W_MMA) {
        // ===================== MMA issuer =====================
        // Per item: S_A(0), S_B(0), then per step j: PV_A(j), S_A(j+1), PV_B(j),
        // S_B(j+1).  S_t(j+1) overwrites the score buffer whose P the PV_t(j) just
        // issued reads: one thread's MMAs run in issue order.  Tile B takes part
        // only when the block has more than 128 query vectors.
        // The whole warp runs the loop (its waits agreed by all lanes); one elected
        // lane -- the same one every time, the lowest, as the warp is converged --
        // issues each group of MMAs and their commits, so that the operand
        // descriptors stay warp-uniform values.
        {
            int32_t g = 0;                     // steps issued (K / V / metadata rings)
            uint32_t n_t[2] = {0, 0};          // steps per tile (s_full / p_full / pv_done phases)
            uint32_t n_q[2] = {0, 0};          // items per tile (q_full phases)
            bool ok = true;
            // Shared-memory descriptors of every operand buffer, built once: the
            // address field is (address >> 4) in the low 14 bits, and every buffer
            // of this CTA lies below 256 KiB, so an offset inside a buffer is added
            // to the descriptor directly.
            const uint64_t dq = tc::sdesc_sw128(sbase + OFF_Q, 16, 1024);          // + t * TILEB
            const uint64_t dk = tc::sdesc_sw128(sbase + OFF_K, 16, 1024);          // + stage * TILEB
            const uint64_t dv = tc::sdesc_sw128(sbase + OFF_V, HALF, 1024);        // + stage * TILEB
            auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, wait_or_fail(bar, parity, fail));
            };
            for (int32_t wi = i0; wi < i1 && ok; ++wi) {
                const ItemInfo it = item_info(a, wi);
                if (it.steps == 0) continue;
                const bool two = a.u.blocks[it.block].n_rows * G > M;
                // Q of each tile: by TMA (qt_full) or written by the softmax threads (q_full)
                uint64_t *qb0 = a.q_tma ? &x.qt_full[0] : &x.q_full[0];
                uint64_t *qb1 = a.q_tma ? &x.qt_full[1] : &x.q_full[1];
                if (!(ok = wait_all(qb0, n_q[0] & 1u))) break;
                ++n_q[0];
                if (two) {
                    if (!(ok = wait_all(qb1, n_q[1] & 1u))) break;
                    ++n_q[1];
                }
                if (!(ok = wait_all(&x.k_full[g % KSTAGES], (uint32_t)(g / KSTAGES) & 1u))) break;
                tc::fence_after();
                if (kvd::elect_one()) {
                    const uint64_t kb0 = dk + (uint64_t)(((g % KSTAGES) * TILEB) >> 4);
                    issue_s8(tmem + COL_S, dq, kb0);
                    tc::commit(&x.s_full[0]);
                    if (two) {
                        issue_s8(tmem + COL_S + 128u, dq + (uint64_t)(TILEB >> 4), kb0);
                        tc::commit(&x.s_full[1]);
                    }
                    tc::commit(&x.k_empty[g % KSTAGES]);
                }
                __syncwarp();
                for (int32_t j = 0; j < it.steps && ok; ++j) {
                    const int32_t gs = g + j;
                    const bool more = j + 1 < it.steps;
                    // V of the step (loaded a step ahead) first, so that only tile A's P
                    // stands between its softmax and PV_A
                    if (!(ok = wait_all(&x.v_full[gs % VSTAGES], (uint32_t)(gs / VSTAGES) & 1u))) break;
                    if (!(ok = wait_all(&x.p_full[0], (n_t[0] + (uint32_t)j) & 1u))) break;
                    tc::fence_after();
                    const uint64_t vb0 = dv + (uint64_t)(((gs % VSTAGES) * TILEB) >> 4);
                    const uint64_t kb1 = dk + (uint64_t)((((gs + 1) % KSTAGES) * TILEB) >> 4);
                    const uint32_t acc = j > 0 ? 1u : 0u;
                    if (kvd::elect_one()) {
                        issue_pv8(tmem + COL_O, tmem + COL_S, vb0, acc);
                        tc::commit(&x.pv_done[0]);
                    }
                    __syncwarp();
                    if (more) {
                        if (!(ok = wait_all(&x.k_full[(gs + 1) % KSTAGES], (uint32_t)((gs + 1) / KSTAGES) & 1u))) break;
                        tc::fence_after();
                        if (kvd::elect_one()) {
                            issue_s8(tmem + COL_S, dq, kb1);
                            tc::commit(&x.s_full[0]);
                        }
                        __syncwarp();
                    }
                    if (two) {
                        if (!(ok = wait_all(&x.p_full[1], (n_t[1] + (uint32_t)j) & 1u))) break;
                        tc::fence_after();
                        if (kvd::elect_one()) {
                            issue_pv8(tmem + COL_O + 128u, tmem + COL_S + 128u, vb0, acc);
                            tc::commit(&x.pv_done[1]);
                            if (more) {
                                issue_s8(tmem + COL_S + 128u, dq + (uint64_t)(TILEB >> 4), kb1);
                                tc::commit(&x.s_full[1]);
                            }
                        }
                        __syncwarp();
                    }
                    if (kvd::elect_one()) {
                        tc::commit(&x.v_empty[gs % VSTAGES]);
                        if (more) tc::commit(&x.k_empty[(gs + 1) % KSTAGES]);
                    }
                    __syncwarp();
                }
                n_t[0] += (uint32_t)it.steps;
                if (two) n_t[1] += (uint32_t)it.steps;
                g += it.steps;
            }
            // all issued MMAs complete before TMEM is released
            if (kvd::elect_one()) {
                tc::commit(&x.spare);
                (void)kvd::mbar_wait_bounded(&x.spare, 0);
            }
            __syncwarp();
        }
    }
    if (a.cluster > 1) {   // this warp's part in the cluster's two meetings (see the softmax warps' end)
        kvd::cluster_sync();
        kvd::cluster_sync();
    }
    } else {
        // register split: the two softmax warpgroups take more registers
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SM_REGS));
        // ============ softmax / epilogue / merge: warps 0-3 tile A, 4-7 tile B ============
        // Thread n of tile t owns TMEM lane n: query vector 128 t + n of the block.
        const int32_t t = warp >> 2;
        const int32_t n = tid & 127;
        const int32_t qv = M * t + n;
        const uint32_t lane_q = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_mine = tmem + lane_q + COL_S + 128u * (uint32_t)t;
        const uint32_t o_mine = tmem + lane_q + COL_O + 128u * (uint32_t)t;
        uint8_t *q_sm = smem + OFF_Q + t * TILEB;
        const int32_t n_all = a.p.n_work[1];
        int32_t g = 0;                         // steps consumed (rings)
        uint32_t n_s = 0;                      // steps of this tile (s_full / p_full / pv_done phases)
        uint32_t n_w = 0;                      // wbar phases
        bool ok = true;
        bool dep_done = false;
        for (int32_t wi = i0; wi < i1 && ok && warp_ok(fail); ++wi) {
            const ItemInfo it = item_info(a, wi);
            const kvi::DevBlock b = a.u.blocks[it.block];
            const int32_t nq = b.n_rows * G;
            const int32_t nitems = a.p.blk_nitems[it.block];
            if (nitems > 1 && a.cluster > 1) {
                // a split piece is its column's last item (the planner makes it so)
                if (wi + 1 != i1) {
                    if (tid == 0) kvd::report(a.err, kvd::DERR_BOUNDS);
                    break;
                }
                mrg_cl = true;
                mrg_nq = nq;
                mrg_row0 = b.row0;
            }
            if (t == 0 || nq > M) {
                // ---------------- this tile has query vectors in the block ----------------
                int32_t row = -1, rpos = 0;
                if (qv < nq) {
                    row = wi == i0 ? a.p.pf_rows[blockIdx.x * PF_M + qv] : a.u.perm[b.row0 + qv / G];
                    rpos = a.u.rows[row].pos;
                }
                const bool live = row >= 0;
                const int32_t h = hk * G + (qv % G);
                if (!dep_done) {   // before the first read of Q and the first write of an output
                    if (live && it.steps > 0 && !a.q_tma) {
                        const __half *qp = a.q + ((int64_t)row * a.n_head + h) * 128;
                        kvd::prefetch_l2(qp);
                        kvd::prefetch_l2(qp + 64);
                    }
                    kvd::pdl_wait();
                    dep_done = true;
                }
                float m_run = -INFINITY, l_run = 0.f;
                if (it.steps > 0) {
                    // ---- Q of the warp's 32 query vectors -> shared memory (the A operand
                    //      of S = Q K^T), 128-byte swizzle.  Each load instruction covers
                    //      two whole rows (16 lanes x 16 bytes each), so the reads are
                    //      coalesced; lane j's row comes from the lane that owns it ----
                    if (!a.q_tma) {   // (else the Q producer loads it)
                        const int32_t wrow = 32 * (warp & 3);
                        uint4 v[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const int32_t jr = 2 * k + (lane >> 4);      // row of the warp
                            const int32_t rj = __shfl_sync(0xffffffffu, row, jr);
                            const int32_t hj = hk * G + ((M * t + wrow + jr) % G);
                            v[k] = rj >= 0 ? __ldg(reinterpret_cast<const uint4 *>(a.q + ((int64_t)rj * a.n_head + hj) * 128) +
                                                   (lane & 15))
                                           : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const uint32_t rr = (uint32_t)(wrow + 2 * k + (lane >> 4));
                            const uint32_t c = (uint32_t)(lane & 15);
                            *reinterpret_cast<uint4 *>(q_sm + (c >> 3) * HALF + kvd::swz128(rr, c & 7u)) = v[k];
                        }
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive(&x.q_full[t]);
                    }
                    for (int32_t j = 0; j < it.steps; ++j, ++g, ++n_s) {
                        ok = __all_sync(0xffffffffu,
                                        wait_or_fail(&x.meta_full[g % MSLOTS], (uint32_t)(g / MSLOTS) & 1u, fail));
                        if (!ok) break;
                        const Meta &mt = x.meta[g % MSLOTS];
                        const bool full = mt.full != 0;
                        // the cells this row sees (sequence, epoch, causal order, window), as
                        // 128 bits, worked out while S is still being computed
                        uint32_t vm[4] = {~0u, ~0u, ~0u, ~0u};
                        if (!live) {
                            vm[0] = vm[1] = vm[2] = vm[3] = 0u;
                        } else if (!full) {
                            const kvd::PosRange rr = kvd::pos_range(a.u.causal, a.u.n_swa, rpos);
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                const int4 *cs = reinterpret_cast<const int4 *>(&mt.cpos[32 * r]);
                                uint32_t pb = 0;
#pragma unroll
                                for (int q4 = 0; q4 < 8; ++q4) {
                                    const int4 cp = cs[q4];
                                    pb |= (kvd::pos_in(rr, cp.x) ? 1u : 0u) << (4 * q4 + 0);
                                    pb |= (kvd::pos_in(rr, cp.y) ? 1u : 0u) << (4 * q4 + 1);
                                    pb |= (kvd::pos_in(rr, cp.z) ? 1u : 0u) << (4 * q4 + 2);
                                    pb |= (kvd::pos_in(rr, cp.w) ? 1u : 0u) << (4 * q4 + 3);
                                }
                                vm[r] = pb & mt.has[r];
                            }
                        }
                        ok = __all_sync(0xffffffffu, wait_or_fail(&x.s_full[t], n_s & 1u, fail));
                        if (!ok) break;
                        tc::fence_after();
                        uint32_t sb[128];
                        tc::ld128(s_mine, sb);
                        if (!live || !full) {
#pragma unroll
                            for (int c = 0; c < 128; ++c)
                                sb[c] = ((vm[c >> 5] >> (c & 31)) & 1u) ? sb[c] : __float_as_uint(-INFINITY);
                        }
                        float mx[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) mx[u] = max3f(-INFINITY, __uint_as_float(sb[2 * u]), __uint_as_float(sb[2 * u + 1]));
#pragma unroll
                        for (int c = 16; c < 128; c += 2)
                            mx[(c >> 1) & 7] = max3f(mx[(c >> 1) & 7], __uint_as_float(sb[c]), __uint_as_float(sb[c + 1]));
                        const float tmax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
                                           a.scale_log2;
                        const float m_new = fmaxf(m_run, tmax);
                        const bool grow = m_new > m_run + RESCALE_LOG2 || (m_run == -INFINITY && m_new != -INFINITY);
                        float alpha = 1.f;
                        if (grow) {
                            alpha = ex2_approx(m_run - m_new);
                            m_run = m_new;
                            l_run *= alpha;
                        }
                        // ---- O *= alpha where the row's running maximum moved (rare): O is
                        //      stable once PV of the previous step finished ----
                        if (j > 0 && __any_sync(0xffffffffu, grow)) {
                            ok = __all_sync(0xffffffffu, wait_or_fail(&x.pv_done[t], (n_s - 1) & 1u, fail));
                            if (!ok) break;
                            tc::fence_after();
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t r[32];
                                tc::ld32(o_mine + 32u * (uint32_t)q, r);
#pragma unroll
                                for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                                tc::st32(o_mine + 32u * (uint32_t)q, r);
                            }
                        }
                        // ---- P = 2^(s*scale - m) as fp16 pairs over the first 64 S columns
                        //      (cell c in column c / 2); the row sum adds those same fp16
                        //      values in fp32 ----
                        {
                            // no maximum yet (nothing visible so far, or a lane past the block):
                            // subtract +inf so that every exponent is -inf and P is 0
                            const float nm = m_run != -INFINITY ? -m_run : -INFINITY;
                            const uint64_t sc2 = pk2(a.scale_log2, a.scale_log2), nm2 = pk2(nm, nm);
                            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh) {
                                uint32_t pw[32];
#pragma unroll
                                for (int c2 = 0; c2 < 32; ++c2) {
                                    const int c = 64 * hh + 2 * c2;
                                    float x0, x1;
                                    upk2(ffma2(pk2(__uint_as_float(sb[c]), __uint_as_float(sb[c + 1])), sc2, nm2), x0,
                                         x1);
                                    const uint32_t p2 = ex2_h2(x0, x1);
                                    pw[c2] = p2;
                                    sum_h2(p2, ls[(c2 & 1) * 2], ls[(c2 & 1) * 2 + 1]);
                                }
                                tc::st32(s_mine + 32u * (uint32_t)hh, pw);
                            }
                            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                        }
                        bool zeroed = false;
                        if (t == 0 && !full) {
                            // V rows of cells nobody in the block sees: zero (P is 0 there; V may
                            // be garbage); thread n clears cell n's row in both d halves
                            ok = __all_sync(0xffffffffu,
                                            wait_or_fail(&x.v_full[g % VSTAGES], (uint32_t)(g / VSTAGES) & 1u, fail));
                            if (!ok) break;
                            if (!((mt.anyvis[n >> 5] >> (n & 31)) & 1u)) {
                                uint8_t *vs = smem + OFF_V + (g % VSTAGES) * TILEB + n * 128;
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    *reinterpret_cast<uint4 *>(vs + c * 16) = make_uint4(0, 0, 0, 0);
                                    *reinterpret_cast<uint4 *>(vs + HALF + c * 16) = make_uint4(0, 0, 0, 0);
                                }
                            }
                            zeroed = true;
                        }
                        tc::wait_st();                     // P (and a rescaled O) are in TMEM
                        if (zeroed) kvd::fence_proxy_async_smem();   // zeroed V rows are visible to the MMA
                        tc::fence_before();
                        kvd::mbar_arrive(&x.p_full[t]);
                    }
                    if (!ok) break;
                    // ---- wait for the item's last PV ----
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.pv_done[t], (n_s - 1) & 1u, fail));
                    if (!ok) break;
                    tc::fence_after();
                }
                // ---- epilogue: the normalised row, or this piece's partial.  Each
                //      32-column quarter of the warp's 32 rows is staged in the warp's own
                //      4 KiB of the tile's Q area (free: the item's last S has completed,
                //      and the next item's Q is written by these same threads after this),
                //      128-byte swizzled.  A partial's rows are consecutive: one TMA store
                //      per quarter writes them (the tensor map undoes the swizzle); an
                //      output row goes out 8 lanes per 128-byte segment ----
                const bool split = nitems > 1;
                if (split && a.cluster > 1) {
                    // ---- a piece of a block split over the cluster: its (m, l) and its
                    //      unnormalised O row stay in this CTA's shared memory, row qv at
                    //      512 qv with the 16-byte chunks XOR-swizzled by qv (conflict-free
                    //      for the writing warp and for a reading warp alike): tile A's
                    //      rows over the Q area, tile B's over the K ring, both idle now ----
                    x.mlx[qv] = make_float2(m_run, l_run);
                    uint8_t *rowp = smem + (uint32_t)qv * 512u;
                    const uint32_t sw = (uint32_t)(qv & 31);
                    if (it.steps > 0) {
#pragma unroll 1
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t ob[64];
                            tc::ld64(o_mine + 64u * (uint32_t)hh, ob);
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                *reinterpret_cast<uint4 *>(rowp + 16u * ((uint32_t)(16 * hh + c) ^ sw)) =
                                    make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) *reinterpret_cast<uint4 *>(rowp + 16u * c) = make_uint4(0, 0, 0, 0);
                    }
                    tc::fence_before();
                    continue;
                }
                float *dst = nullptr;
                float sc = 1.f;
                const int64_t prow = ((int64_t)wi * a.n_head_kv + hk) * PF_M;   // this item's first partial row
                if (!split) {
                    if (live) dst = a.o + ((int64_t)row * a.n_head + h) * 128;
                    sc = l_run > 0.f ? 1.f / l_run : 0.f;
                } else {
                    *reinterpret_cast<float2 *>(a.part_ml + (prow + qv) * 2) = make_float2(m_run, l_run);
                }
                if (it.steps > 0) {
                // the O row in two TMEM reads of 64 columns (warp collective)
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                uint32_t ob[64];
                tc::ld64(o_mine + 64u * (uint32_t)hh, ob);
#pragma unroll
                for (int qh = 0; qh < 2; ++qh) {
                    const int q = 2 * hh + qh;
                    // two staging buffers per warp (its rows in either d half of the tile's
                    // Q area), used in turn: a partial's TMA store of one overlaps the
                    // staging of the next
                    uint8_t *stg = q_sm + qh * HALF + 4096 * (warp & 3);
                    if (split && lane == 0 && q >= 2) kvd::bulk_wait_read<1>();   // the store from this buffer has read it
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4 *>(stg + kvd::swz128((uint32_t)lane, (uint32_t)c)) =
                            make_float4(__uint_as_float(ob[32 * qh + 4 * c]) * sc, __uint_as_float(ob[32 * qh + 4 * c + 1]) * sc,
                                        __uint_as_float(ob[32 * qh + 4 * c + 2]) * sc,
                                        __uint_as_float(ob[32 * qh + 4 * c + 3]) * sc);
                    if (split) {
                        kvd::fence_proxy_async_smem();   // the staged rows are visible to the TMA store
                        __syncwarp();
                        if (lane == 0) {
                            kvd::tma_store_2d(&tm_part, 32 * q, (int32_t)(prow + M * t + 32 * (warp & 3)), stg);
                            kvd::bulk_commit();
                        }
                        __syncwarp();
                    } else {
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int32_t jr = 4 * k + (lane >> 3);         // row of the warp
                            const uint32_t c = (uint32_t)(lane & 7);
                            float *dj = reinterpret_cast<float *>(
                                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), jr));
                            if (dj)
                                *reinterpret_cast<float4 *>(dj + 32 * q + 4 * c) =
                                    *reinterpret_cast<const float4 *>(stg + kvd::swz128((uint32_t)jr, c));
                        }
                        __syncwarp();
                    }
                }
                }
                if (split && lane == 0) {
                    // the partial's rows are written before the piece is counted
                    kvd::bulk_wait_all();
                    kvd::fence_proxy_async_global();
                }
                if (a.q_tma) {
                    // the Q area is free for the next item's Q (TMA writes after these
                    // generic accesses)
                    kvd::fence_proxy_async_smem();
                    kvd::mbar_arrive(&x.q_free[t]);
                }
                } else if (dst) {
                    // a block that sees nothing (a single item, no step): zeros, written
                    // directly (the Q area may already hold the next item's Q)
#pragma unroll
                    for (int c = 0; c < 32; ++c) *reinterpret_cast<float4 *>(dst + 4 * c) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                tc::fence_before();
            } else {
                g += it.steps;                     // tile B has no query vector in this block
            }
            if (nitems == 1 || a.cluster > 1) continue;
            // ---------------- a piece of a split block ----------------
            // All 256 softmax threads meet once the piece's rows are written (every
            // thread waits, so none can arrive for a later phase early); thread 0
            // then counts the piece.  The CTAs whose last item is a piece of this
            // block wait until all pieces are counted and merge a share each.
            if (!dep_done) {
                kvd::pdl_wait();
                dep_done = true;
            }
            kvd::fence_proxy_async_smem();   // the staging writes come before any later bulk copy into it
            kvd::mbar_arrive(&x.wbar);
            ok = __all_sync(0xffffffffu, wait_or_fail(&x.wbar, n_w & 1u, fail));
            ++n_w;
            if (!ok) break;
            const bool mine = wi + 1 == i1;
            int32_t *cnt = a.p.counters + (int64_t)it.block * a.n_head_kv + hk;
            const int32_t it0 = a.p.blk_item0[it.block] - a.p.cap_dec;
            // The merge participants are the block's pieces that are the last item of
            // their column, in item order: warp 0 finds them with one ballot per 32
            // pieces (np of them, `rank` of them before mine).
            int32_t np = 0, rank = 0;
            if (warp == 0 && mine) {
                for (int32_t k0 = it0; k0 < it0 + nitems; k0 += 32) {
                    const int32_t k = k0 + lane;
                    const bool part = k < it0 + nitems && last_of_column(a, k, n_all);
                    const uint32_t bal = __ballot_sync(0xffffffffu, part);
                    np += __popc(bal);
                    rank += __popc(bal & __ballot_sync(0xffffffffu, k < wi));
                }
            }
            // The merge of query vectors mrg_lo .. mrg_hi - 1:
            //   O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q.
            // Each piece's O rows of a share are one contiguous range, and so are their
            // (m, l): two bulk copies per piece bring them into shared memory (the Q area
            // and the K/V rings, idle now), in passes of rp query vectors.
            const int64_t istride = (int64_t)a.n_head_kv * PF_M;           // partial rows per item
            const int64_t prow0 = ((int64_t)it0 * a.n_head_kv + hk) * PF_M;
            constexpr uint32_t ROWB = 128 * 4;                           // bytes of one O row
            constexpr uint32_t MCAP = OFF_AUX;                           // shared bytes free for the merge
            // rows per pass: a multiple of 8, with room for one more (m, l) per piece
            const int32_t rp = min(PF_M, (int32_t)(((MCAP / (uint32_t)nitems - 8u) / (ROWB + 8u)) & ~7u));
            auto issue_pass = [&](int32_t v0, int32_t R) {   // one thread: the copies of one pass
                const int32_t R2 = (R + 1) & ~1;                         // (m, l) rows copied: an even count
                const uint32_t qstride = (uint32_t)R * ROWB;
                float2 *mls = reinterpret_cast<float2 *>(smem + (uint32_t)nitems * qstride);   // [piece][R2]
                kvd::fence_proxy_async_global();
                kvd::mbar_arrive_expect_tx(&x.mbar, (uint32_t)nitems * (qstride + 8u * (uint32_t)R2));
                for (int32_t q = 0; q < nitems; ++q) {
                    const int64_t r0 = prow0 + q * istride + v0;
                    kvd::bulk_load(mls + q * R2, reinterpret_cast<const float2 *>(a.part_ml) + r0, 8u * (uint32_t)R2,
                                   &x.mbar);
                    kvd::bulk_load(smem + (uint32_t)q * qstride, a.part + r0 * 128, qstride, &x.mbar);
                }
            };
            if (warp == 0) {
                if (lane == 0) {
                    // count the piece: every thread's writes of it came before the barrier
                    // above, so one release by this thread publishes them all
                    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
                    if (mine) {
                        // wait (bounded) until every piece of the block is counted
                        long long t0c = clock64();
                        while (ld_acquire(cnt) < nitems) {
                            if (*fail || clock64() - t0c > kvd::WAIT_LIMIT_CYCLES) {
                                *fail = 1;
                                break;
                            }
                            __nanosleep(64);
                        }
                        // shares start on a multiple of 8 query vectors (16-byte aligned
                        // (m, l) copies)
                        const int32_t lo = (int32_t)((int64_t)nq * rank / np) & ~7;
                        const int32_t hi = rank + 1 == np ? nq : (int32_t)((int64_t)nq * (rank + 1) / np) & ~7;
                        x.mrg_lo = lo;
                        x.mrg_hi = hi;
                        // the first pass's copies go out before the other warps are woken
                        if (lo < hi && rp >= 8 && !*fail) issue_pass(lo, min(rp, hi - lo));
                    }
                }
                // the rest of warp 0 waits here, not on the barrier below: lane 0 is
                // the one that completes it
                __syncwarp();
                if (mine && lane == 0) kvd::mbar_arrive(&x.gbar);
            }
            if (!mine) continue;
            if (warp != 0) ok = __all_sync(0xffffffffu, wait_or_fail(&x.gbar, 0, fail));
            if (!ok || !warp_ok(fail)) break;
            if (rp < 8) {
                if (tid == 0) kvd::report(a.err, kvd::DERR_BOUNDS);
                break;
            }
            // ---- a pass: the weights from the (m, l) (a thread per query vector), then
            //      the rows summed piece by piece as they land and stored, 512 contiguous
            //      bytes each ----
            {
                const int32_t lo = x.mrg_lo, hi = x.mrg_hi;
                uint32_t n_m = 0;                                          // mbar phases
                for (int32_t v0 = lo; v0 < hi; v0 += rp, ++n_m) {
                    const int32_t R = min(rp, hi - v0);
                    const int32_t R2 = (R + 1) & ~1;
                    const uint32_t qstride = (uint32_t)R * ROWB;
                    float2 *mls = reinterpret_cast<float2 *>(smem + (uint32_t)nitems * qstride);
                    if (v0 != lo && tid == 0) issue_pass(v0, R);
                    // warp w's output rows, one load per lane (lane 8k + r: query vector
                    // v0 + 64k + 8w + r), before they are needed
                    int32_t orow = -1;
                    {
                        const int32_t vl = v0 + 64 * (lane >> 3) + 8 * warp + (lane & 7);
                        if (vl < v0 + R) orow = a.u.perm[b.row0 + vl / G];
                    }
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.mbar, n_m & 1u, fail));   // rows and (m, l) landed
                    if (!ok) break;
                    // pass 1, a thread per query vector: the pieces' weights 2^(m_q - M) / L
                    // replace their m in shared memory
                    for (int32_t r = tid; r < R; r += NSM) {
                        if (nitems <= 8) {
                            float2 ml[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q) ml[q] = q < nitems ? mls[q * R2 + r] : make_float2(-INFINITY, 0.f);
                            float Mx = -INFINITY;
#pragma unroll
                            for (int q = 0; q < 8; ++q) Mx = fmaxf(Mx, ml[q].x);
                            float w[8], L = 0.f;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                w[q] = (ml[q].x == -INFINITY || Mx == -INFINITY) ? 0.f : ex2_approx(ml[q].x - Mx);
                                L = fmaf(ml[q].y, w[q], L);
                            }
                            const float inv = L > 0.f ? rcp_approx(L) : 0.f;
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                if (q < nitems) mls[q * R2 + r].x = w[q] * inv;
                        } else {
                            float Mx = -INFINITY;
                            for (int32_t q = 0; q < nitems; ++q) Mx = fmaxf(Mx, mls[q * R2 + r].x);
                            float L = 0.f;
                            for (int32_t q = 0; q < nitems; ++q) {
                                const float2 ml = mls[q * R2 + r];
                                const float w = (ml.x == -INFINITY || Mx == -INFINITY) ? 0.f : ex2_approx(ml.x - Mx);
                                L = fmaf(ml.y, w, L);
                                mls[q * R2 + r].x = w;
                            }
                            const float inv = L > 0.f ? rcp_approx(L) : 0.f;
                            for (int32_t q = 0; q < nitems; ++q) mls[q * R2 + r].x *= inv;
                        }
                    }
                    kvd::mbar_arrive(&x.wbar);                             // the weights are in place
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.wbar, n_w & 1u, fail));
                    ++n_w;
                    if (!ok) break;
                    // pass 2, a warp per 8 query vectors at once (v0 + 64k + 8w + r), lane l
                    // owning d = 4l .. 4l + 3
                    for (int32_t k = 0; 64 * k + 8 * warp < R && ok; ++k) {
                        const int32_t rb = 64 * k + 8 * warp;          // first row of the batch (pass-relative)
                        const int32_t nr = min(8, R - rb);
                        float4 acc[8];
#pragma unroll
                        for (int r = 0; r < 8; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int32_t q = 0; q < nitems; ++q) {
                            float w[8];
                            float4 ov[8];
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                w[r] = r < nr ? mls[q * R2 + rb + r].x : 0.f;
                                ov[r] = r < nr ? *reinterpret_cast<const float4 *>(smem + (uint32_t)q * qstride +
                                                                                   (uint32_t)(rb + r) * ROWB + 16 * lane)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                            }
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                acc[r].x = fmaf(ov[r].x, w[r], acc[r].x);
                                acc[r].y = fmaf(ov[r].y, w[r], acc[r].y);
                                acc[r].z = fmaf(ov[r].z, w[r], acc[r].z);
                                acc[r].w = fmaf(ov[r].w, w[r], acc[r].w);
                            }
                        }
                        if (!ok) break;
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            const int32_t mrow = __shfl_sync(0xffffffffu, orow, 8 * k + r);
                            if (r < nr) {
                                const int32_t v = v0 + rb + r;
                                *reinterpret_cast<float4 *>(a.o + ((int64_t)mrow * a.n_head + hk * G + (v % G)) * 128 +
                                                            4 * lane) = acc[r];
                            }
                        }
                    }
                    if (!ok) break;
                    if (v0 + rp < hi) {
                        // every read of this pass is done before the next pass's copies land
                        kvd::fence_proxy_async_smem();
                        kvd::mbar_arrive(&x.wbar);
                        ok = __all_sync(0xffffffffu, wait_or_fail(&x.wbar, n_w & 1u, fail));
                        ++n_w;
                        if (!ok) break;
                    }
                }
                if (!ok) break;
            }
            // done reading the partials: count again; the arrival that completes the
            // count (every piece once, every participant once more) resets it for the
            // next launch
            kvd::mbar_arrive(&x.wbar);
            if (tid == 0 && wait_or_fail(&x.wbar, n_w & 1u, fail)) {
                if (atomicAdd(cnt, 1) == nitems + np - 1) atomicExch(cnt, 0);
            }
            ++n_w;
        }
        if (a.cluster > 1) {
            // Every thread of every CTA of the cluster reaches both barriers exactly once,
            // after its bounded work: the first makes the staged pieces visible across the
            // cluster, the second keeps each CTA's shared memory alive until the others
            // have read it.
            kvd::cluster_sync();
            if (warp < 8 && mrg_cl && warp_ok(fail)) {
                // ---- merge query vectors lo .. hi - 1 of the split block, this CTA's
                //      share by its rank in the cluster:
                //      O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q over the C pieces,
                //      read from the pieces' shared memory, lane l owning d = 4l .. 4l + 3 ----
                constexpr int C = kvi::PF_CLUSTER;       // the launch's cluster size (checked at launch)
                const uint32_t rank = kvd::cluster_ctarank();
                const int32_t lo = (int32_t)((int64_t)mrg_nq * rank / C), hi = (int32_t)((int64_t)mrg_nq * (rank + 1) / C);
                uint32_t ob_q[C], ml_q[C];
#pragma unroll
                for (int q = 0; q < C; ++q) {
                    ob_q[q] = kvd::map_cluster(sbase, (uint32_t)q);
                    ml_q[q] = kvd::map_cluster(kvd::smem_u32(&x.mlx[0]), (uint32_t)q);
                }
                // Warp w takes vectors lo + 32k + 4w + r, r = 0..3, four at once: lane
                // 4r + q reads piece q's (m, l) of vector r (one load each), the weights
                // come from shuffles, and each lane then reads its d slice of the 16
                // rows (4 vectors x 4 pieces) in one round of loads.
                const int32_t rr = lane >> 2, qq = lane & 3;
                for (int32_t v0 = lo + 4 * warp; v0 < hi; v0 += 32) {
                    const int32_t vr = v0 + rr;
                    float2 ml = make_float2(-INFINITY, 0.f);
                    if (vr < hi) ml = kvd::ld_cluster_f2(ml_q[qq] + 8u * (uint32_t)vr);
                    float4 o4[4][C];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int32_t v = min(v0 + r, hi - 1);
                        const uint32_t off = (uint32_t)v * 512u + 16u * ((uint32_t)lane ^ (uint32_t)(v & 31));
#pragma unroll
                        for (int q = 0; q < C; ++q) o4[r][q] = kvd::ld_cluster_f4(ob_q[q] + off);
                    }
                    float Mx = fmaxf(ml.x, __shfl_xor_sync(0xffffffffu, ml.x, 1));
                    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, 2));
                    const float w = (ml.x == -INFINITY || Mx == -INFINITY) ? 0.f : ex2_approx(ml.x - Mx);
                    float L = ml.y * w;
                    L += __shfl_xor_sync(0xffffffffu, L, 1);
                    L += __shfl_xor_sync(0xffffffffu, L, 2);
                    const float wn = L > 0.f ? w * rcp_approx(L) : 0.f;   // piece qq's weight for vector rr
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int q = 0; q < C; ++q) {
                            const float wq = __shfl_sync(0xffffffffu, wn, 4 * r + q);
                            acc.x = fmaf(o4[r][q].x, wq, acc.x);
                            acc.y = fmaf(o4[r][q].y, wq, acc.y);
                            acc.z = fmaf(o4[r][q].z, wq, acc.z);
                            acc.w = fmaf(o4[r][q].w, wq, acc.w);
                        }
                        const int32_t v = v0 + r;
                        if (v < hi) {
                            const int32_t row = a.u.perm[mrg_row0 + v / G];
                            *reinterpret_cast<float4 *>(a.o + ((int64_t)row * a.n_head + hk * G + (v % G)) * 128 + 4 * lane) =
                                acc;
                        }
                    }
                }
            }
            kvd::cluster_sync();
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
    if (*fail && tid == 0) kvd::report(a.err, kvd::DERR_MMA_TIMEOUT);
}

}  // namespace

namespace kvk {

cudaError_t load_prefill_kernels() {
    cudaError_t e = cudaFuncSetAttribute(k_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // clusters of up to 8 CTAs are portable; none larger is asked for
    return cudaFuncSetAttribute(k_prefill, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
}

// Clusters of `cluster` attention CTAs that can be resident at once on the current
// device (0: the launch would fail, or the query did).
int prefill_max_active_clusters(int cluster) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster, 1);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void *)k_prefill, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// The shared-memory attribute was set for the current device by load_prefill_kernels.
cudaError_t launch_prefill(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const CUtensorMap *tm_part,
                           const CUtensorMap *tm_q, const PrefillArgs &a, int32_t grid_x, cudaStream_t st) {
    // A programmatic dependent of the kernel before it: the attention kernel sets
    // up (and, with early_ok, reads its plan) while the K/V store finishes.
    // With a.cluster > 1, also a thread-block cluster of that many columns (the grid's
    // column count is a multiple of it).
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)(a.cluster > 1 ? a.cluster : 1);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    if (a.cluster != 1 && (a.cluster != kvi::PF_CLUSTER || grid_x % a.cluster != 0)) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, a.n_head_kv);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = a.cluster > 1 ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_prefill, *tm_k, *tm_v, *tm_part, *tm_q, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kvk
