// K3b: GQA flash attention, prefill / mixed path, on tcgen05 tensor cores.
//
// "llama.cpp and the ubatch", "Chunked prefill is the same mechanism": a
// chunk of U rows against C cached cells is a [U, C+U] score matrix; with the
// mask of "The mask is doing the work" (occupied, same first sequence id,
// not later) it is the same softmax(q K^T / sqrt(d) + mask) V as decode, but
// now a dense contraction worth putting on the tensor cores.
//
// Design (sm_103a, one CTA of 192 threads per SM):
//  * a block = up to 128 query vectors (rows sharing a stream and first
//    sequence id, times the GQA group) = the 128 TMEM lanes of one MMA tile;
//    a work item = one block, one KV head, a chunk of the block's list of
//    visible 64-cell tiles, consumed two at a time (N = 128 cells);
//  * warp 4 (one thread) streams K and V tiles with TMA (128-byte swizzle)
//    into a 2-stage ring; warp 5 allocates TMEM and one thread issues
//    tcgen05.mma: S = Q K^T (M 128, N 128, K 128) into one of two TMEM score
//    buffers, then O += P V (K = 128 cells, V read MN-major) into a TMEM
//    accumulator; tcgen05.commit signals the mbarriers;
//  * warps 0-3 (thread = TMEM lane = query vector) read S with tcgen05.ld,
//    apply the mask per cell on tiles that are not fully visible, run the
//    online softmax in base 2, write P (fp16) to shared memory in the
//    swizzled K-major layout, and rescale O in TMEM only when the running
//    maximum grew by more than 2^8 (otherwise the stale maximum is kept; the
//    final normalisation uses the same one);
//  * cells nobody in the block may see get their V rows zeroed in shared
//    memory before the PV product (P is 0 there, but 0 * NaN would not be);
//  * split-K chunks of one block are merged by the last CTA to finish, as in
//    the decode path; every mbarrier wait is bounded.

#include "dev_common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace {

using kvi::TILE;

constexpr int NT = 192;
constexpr int M = 128;
constexpr int HALF = 128 * 128;          // [128 rows][64 fp16], 128-byte rows
constexpr int TILEB = 2 * HALF;          // 32 KiB
constexpr int BOX = 64 * 128;            // one TMA box: 64 rows x 64 fp16
constexpr int STAGES = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_P = OFF_Q + TILEB;
constexpr int OFF_K = OFF_P + TILEB;
constexpr int OFF_V = OFF_K + STAGES * TILEB;
constexpr int OFF_AUX = OFF_V + STAGES * TILEB;
constexpr int PART_STRIDE = 132;
constexpr uint32_t TMEM_COLS = 512;      // S0 [0,128), S1 [128,256), O [256,384)
constexpr uint32_t COL_O = 256;
constexpr float RESCALE_LOG2 = 8.0f;

constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16(128, 128, 0, 1);

struct Meta {                 // per stage: what the producer learned about the pair tile
    int32_t full;
    int32_t pad[3];
    int32_t cpos[128];
    uint8_t has[128];         // cell holds the block's sequence and is not from a later ubatch
    uint8_t anyvis[128];      // ... and some row of the block may see it
};

struct ItemSlot {             // per work item: the query vector behind each TMEM lane
    int32_t row[M];           // ubatch row, -1 for lanes past the block's query vectors
    int32_t rpos[M];
};

struct __align__(16) Aux {
    uint64_t k_full[STAGES], v_full[STAGES], kv_empty[STAGES];
    uint64_t s_full[2], p_full, pv_done, q_full, spare;
    uint32_t tmem_base;
    int32_t fail;
    int32_t flag;
    int32_t pad;
    Meta meta[STAGES];
    ItemSlot islot[2];
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
            kvd::mbar_init(&x.k_full[s], 33);   // lane 0's expect_tx + 32 producer lanes
            kvd::mbar_init(&x.v_full[s], 1);
            kvd::mbar_init(&x.kv_empty[s], 1);
        }
        kvd::mbar_init(&x.s_full[0], 1);
        kvd::mbar_init(&x.s_full[1], 1);
        kvd::mbar_init(&x.p_full, 128);
        kvd::mbar_init(&x.pv_done, 1);
        kvd::mbar_init(&x.q_full, 128);
        kvd::mbar_init(&x.spare, 1);
        x.fail = 0;
        kvd::fence_mbar_init();
    }
    if (warp == 5) {
        tc::alloc(&x.tmem_base, TMEM_COLS);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = x.tmem_base;

    if (warp == 4) {
        // ===================== producer (whole warp) =====================
        const int32_t lane = tid & 31;
        int32_t issued = 0, nonempty = 0;
        for (int32_t wi = i0; wi < i1 && warp_ok(fail); ++wi) {
            const ItemInfo it = item_info(a, wi);
            if (it.pairs == 0) continue;
            const kvi::DevBlock b = a.u.blocks[it.block];
            const int32_t nqv = b.n_rows * G;
            ItemSlot &is = x.islot[nonempty & 1];
            ++nonempty;
            const int32_t *list = a.p.tiles + (int64_t)it.block * a.p.tile_stride;
            const uint32_t *flg = a.p.flags + (int64_t)it.block * a.p.tile_stride;
            for (int32_t j = 0; j < it.pairs; ++j) {
                const int32_t st = issued % STAGES;
                // everything this pair needs from global memory, fetched before the
                // stage is free so that only the TMA issue waits for it
                int32_t tt[2];
                bool fullh[2];
                for (int h = 0; h < 2; ++h) {
                    const int32_t e = it.t0 + 2 * j + h;
                    tt[h] = e < it.t1 ? list[e] : -1;
                    fullh[h] = tt[h] >= 0 && (int32_t)(flg[tt[h]] & 0xffffu) == b.n_rows * TILE;
                }
                const bool full = fullh[0] && fullh[1];
                bool mhas[4], many[4];
                int32_t mpos[4];
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
                                const int64_t g = (int64_t)b.stream * a.u.kv_size + jc;
                                const uint64_t w = a.u.cell_bits[g * a.u.n_words + (b.seq0 >> 6)];
                                has = ((w >> (b.seq0 & 63)) & 1ull) && a.u.cell_epoch[g] <= a.u.ub_epoch;
                                cp = a.u.cell_pos[g];
                            }
                        }
                        mhas[r] = has;
                        mpos[r] = cp;
                        many[r] = has && (!a.u.causal || cp <= b.pos_max);
                    }
                }
                int32_t lrow[4], lpos[4];
                if (j == 0) {
                    for (int r = 0; r < 4; ++r) {
                        const int32_t n = lane + 32 * r;
                        lrow[r] = -1;
                        lpos[r] = 0;
                        if (n < nqv) {
                            lrow[r] = a.u.perm[b.row0 + n / G];
                            lpos[r] = a.u.rows[lrow[r]].pos;
                        }
                    }
                }
                if (issued >= STAGES &&
                    !__all_sync(0xffffffffu,
                                wait_or_fail(&x.kv_empty[st], (uint32_t)((issued / STAGES) - 1) & 1u, fail)))
                    break;
                if (j == 0) {
                    // the item's lane table; the slot's previous reader started two or more
                    // loads ago, and this load's stage was just released, so it is done with it
                    for (int r = 0; r < 4; ++r) {
                        is.row[lane + 32 * r] = lrow[r];
                        is.rpos[lane + 32 * r] = lpos[r];
                    }
                }
                Meta &mt = x.meta[st];
                if (lane == 0) {
                    int32_t ys[2];
                    for (int h = 0; h < 2; ++h)   // a missing second tile: out of bounds, TMA writes zeros
                        ys[h] = tt[h] >= 0 ? b.stream * a.u.kv_size + tt[h] * TILE : -TILE;
                    uint8_t *ks = smem + OFF_K + st * TILEB;
                    uint8_t *vs = smem + OFF_V + st * TILEB;
                    const int32_t xk = hk * 128;
                    kvd::fence_proxy_async_smem();
                    kvd::mbar_arrive_expect_tx(&x.k_full[st], TILEB);
                    for (int h = 0; h < 2; ++h) {
                        kvd::tma_load_2d(ks + h * BOX, &tm_k, xk, ys[h], &x.k_full[st]);
                        kvd::tma_load_2d(ks + HALF + h * BOX, &tm_k, xk + 64, ys[h], &x.k_full[st]);
                    }
                    kvd::mbar_arrive_expect_tx(&x.v_full[st], TILEB);
                    for (int h = 0; h < 2; ++h) {
                        kvd::tma_load_2d(vs + h * BOX, &tm_v, xk, ys[h], &x.v_full[st]);
                        kvd::tma_load_2d(vs + HALF + h * BOX, &tm_v, xk + 64, ys[h], &x.v_full[st]);
                    }
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
                kvd::mbar_arrive(&x.k_full[st]);
                ++issued;
            }
        }
        if (*fail && lane == 0) {
            // let loads already issued land before the CTA exits
            for (int32_t q = issued > STAGES ? issued - STAGES : 0; q < issued; ++q) {
                (void)kvd::mbar_wait_bounded(&x.k_full[q % STAGES], (uint32_t)(q / STAGES) & 1u);
                (void)kvd::mbar_wait_bounded(&x.v_full[q % STAGES], (uint32_t)(q / STAGES) & 1u);
            }
        }
    } else if (warp == 5) {
        // ===================== MMA issuer =====================
        if ((tid & 31) == 0) {
            int32_t gidx = 0;          // global pair-tile counter (stage ring)
            uint32_t n_q = 0, n_p = 0;
            uint32_t n_s[2] = {0, 0};
            const uint32_t q_addr = sbase + OFF_Q;
            const uint32_t p_addr = sbase + OFF_P;
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
            };
            for (int32_t wi = i0; wi < i1 && !*fail; ++wi) {
                const ItemInfo it = item_info(a, wi);
                if (it.pairs == 0) continue;
                if (!wait_or_fail(&x.q_full, n_q & 1u, fail)) break;
                ++n_q;
                tc::fence_after();
                bool ok = true;
                for (int32_t j = 0; j < 2 && j < it.pairs && ok; ++j) {
                    const int32_t gi = gidx + j;
                    ok = wait_or_fail(&x.k_full[gi % STAGES], (uint32_t)(gi / STAGES) & 1u, fail);
                    if (ok) { tc::fence_after(); issue_s(gi, j & 1); ++n_s[j & 1]; }
                }
                for (int32_t j = 0; j < it.pairs && ok; ++j) {
                    const int32_t gi = gidx + j;
                    ok = wait_or_fail(&x.p_full, n_p & 1u, fail);
                    if (!ok) break;
                    ++n_p;
                    ok = wait_or_fail(&x.v_full[gi % STAGES], (uint32_t)(gi / STAGES) & 1u, fail);
                    if (!ok) break;
                    tc::fence_after();
                    const uint32_t v_addr = sbase + OFF_V + (gi % STAGES) * TILEB;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t aoff = (uint32_t)(kk >> 2) * HALF + (uint32_t)(kk & 3) * 32u;
                        const uint32_t boff = (uint32_t)kk * 2048u;
                        tc::mma_ss(tmem + COL_O, tc::sdesc_sw128(p_addr + aoff, 16, 1024),
                                   tc::sdesc_sw128(v_addr + boff, HALF, 1024), IDESC_PV,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(&x.pv_done);
                    tc::commit(&x.kv_empty[gi % STAGES]);
                    if (j + 2 < it.pairs) {
                        const int32_t g2 = gi + 2;
                        ok = wait_or_fail(&x.k_full[g2 % STAGES], (uint32_t)(g2 / STAGES) & 1u, fail);
                        if (ok) { tc::fence_after(); issue_s(g2, j & 1); ++n_s[j & 1]; }
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
        // ===================== softmax / correction / epilogue (warps 0-3) =====================
        const int32_t n = tid;                 // TMEM lane = query vector
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t n_s[2] = {0, 0};
        uint32_t n_pv = 0;
        int32_t k = 0;                         // pair tiles consumed (stage ring position)
        int32_t nonempty = 0;
        bool ok = true;
        for (int32_t wi = i0; wi < i1 && ok && warp_ok(fail); ++wi) {
            const ItemInfo it = item_info(a, wi);
            int32_t row = -1, rpos = 0;
            if (it.pairs == 0) {
                // an empty item (its block sees no cell): zeros, or an empty partial
                const kvi::DevBlock b = a.u.blocks[it.block];
                if (n < b.n_rows * G) row = a.u.perm[b.row0 + n / G];
            } else {
                // the first pair's arrival also publishes this item's lane table
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.k_full[k % STAGES], (uint32_t)(k / STAGES) & 1u, fail));
                if (!ok) break;
                const ItemSlot &is = x.islot[nonempty & 1];
                ++nonempty;
                row = is.row[n];
                rpos = is.rpos[n];
            }
            const bool live = row >= 0;
            const int32_t h = hk * G + (n % G);
            float *orow = a.o + ((int64_t)(live ? row : 0) * a.n_head + h) * 128;
            float m_run = -INFINITY, l_run = 0.f;
            float ov[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) ov[c] = 0.f;
            if (it.pairs > 0) {
            // ---- Q tile: row n, 128-byte swizzle, two d-halves ----
            {
                uint8_t *qs = smem + OFF_Q;
                const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((int64_t)(live ? row : 0) * a.n_head + h) * 128);
                uint4 qv[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) qv[c] = live ? src[c] : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4 *>(qs + (c >> 3) * HALF + kvd::swz128(n, c & 7)) = qv[c];
                kvd::fence_proxy_async_smem();
                kvd::mbar_arrive(&x.q_full);
            }
            for (int32_t j = 0; j < it.pairs; ++j, ++k) {
                const int32_t st = k % STAGES;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.k_full[st], (uint32_t)(k / STAGES) & 1u, fail));
                if (!ok) break;
                const Meta &mt = x.meta[st];
                const bool full = mt.full != 0;
                ok = __all_sync(0xffffffffu, wait_or_fail(&x.s_full[j & 1], n_s[j & 1] & 1u, fail));
                if (!ok) break;
                ++n_s[j & 1];
                tc::fence_after();
                // ---- S row -> 128 registers, read from TMEM once, right when it is ready
                //      (TMEM reads stall while the next MMA runs, so pass 2 must not go
                //      back to TMEM); masked cells become -inf; row max in 4 chains ----
                uint32_t sb[128];
                tc::ld128(lane_base + (uint32_t)(j & 1) * 128u, sb);   // warp collective
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (!live) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) sb[c] = __float_as_uint(-INFINITY);
                } else if (!full) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const bool vis = mt.has[c] && (!a.u.causal || mt.cpos[c] <= rpos);
                        if (!vis) sb[c] = __float_as_uint(-INFINITY);
                    }
                }
#pragma unroll
                for (int c = 0; c < 128; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(sb[c]));
                const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.scale_log2;
                const float m_new = fmaxf(m_run, tmax);
                const bool grow = m_new > m_run + RESCALE_LOG2 || (m_run == -INFINITY && m_new != -INFINITY);
                float alpha = 1.f;
                if (grow) {
                    alpha = ex2_approx(m_run - m_new);
                    m_run = m_new;
                    l_run *= alpha;
                }
                // ---- P buffer free and O stable once the previous PV finished ----
                if (j > 0) {
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.pv_done, n_pv & 1u, fail));
                    if (!ok) break;
                    ++n_pv;
                    tc::fence_after();
                }
                // ---- pass 2 (from registers): P = 2^(s*scale - m) as fp16, straight to
                //      shared memory (128-byte swizzled K-major); one exponential in four
                //      on the FMA pipe, the rest on the MUFU unit; row sum in 4 chains ----
                {
                    uint8_t *ps = smem + OFF_P;
                    const bool any = m_run != -INFINITY;   // false for lanes past the block
                    const float nm = -m_run;
                    const float sc = a.scale_log2;
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int c8 = 0; c8 < 16; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = c8 * 8 + 2 * e;
                            const float x0 = fmaf(__uint_as_float(sb[c]), sc, nm);
                            const float x1 = fmaf(__uint_as_float(sb[c + 1]), sc, nm);
                            float p0 = ex2_approx(x0);
                            float p1 = (e & 1) ? ex2_poly(x1) : ex2_approx(x1);
                            p0 = any ? p0 : 0.f;
                            p1 = any ? p1 : 0.f;
                            ls[e] += p0 + p1;
                            __half2 hv = __floats2half2_rn(p0, p1);
                            w[e] = *reinterpret_cast<uint32_t *>(&hv);
                        }
                        *reinterpret_cast<uint4 *>(ps + (c8 >> 3) * HALF + kvd::swz128(n, c8 & 7)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                }
                // ---- O *= alpha where the running maximum moved (rare); O is stable
                //      since the previous PV finished, and this pair's PV waits for us ----
                if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t r[32];
                        const uint32_t ta = lane_base + COL_O + (uint32_t)q4 * 32u;
                        tc::ld32(ta, r);
#pragma unroll
                        for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                        tc::st32(ta, r);
                    }
                    tc::wait_st();
                }
                if (!full) {
                    // V rows of cells nobody in the block sees: zero (P is 0 there; V may be garbage)
                    ok = __all_sync(0xffffffffu, wait_or_fail(&x.v_full[st], (uint32_t)(k / STAGES) & 1u, fail));
                    if (!ok) break;
                    if (!mt.anyvis[n]) {
                        uint8_t *vs = smem + OFF_V + st * TILEB;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4 *>(vs + hh * HALF + n * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                kvd::fence_proxy_async_smem();
                tc::fence_before();
                kvd::mbar_arrive(&x.p_full);
            }
            if (!ok) break;
            // ---- epilogue: wait for the last PV, read O ----
            ok = __all_sync(0xffffffffu, wait_or_fail(&x.pv_done, n_pv & 1u, fail));
            if (!ok) break;
            ++n_pv;
            tc::fence_after();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t r[32];
                tc::ld32(lane_base + COL_O + (uint32_t)q4 * 32u, r);
#pragma unroll
                for (int c = 0; c < 32; ++c) ov[q4 * 32 + c] = __uint_as_float(r[c]);
            }
            tc::fence_before();
            }   // it.pairs > 0
            if (it.nitems == 1) {
                if (live) {
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
                    for (int c = 0; c < 128; c += 4)
                        *reinterpret_cast<float4 *>(orow + c) =
                            make_float4(ov[c] * inv, ov[c + 1] * inv, ov[c + 2] * inv, ov[c + 3] * inv);
                }
            } else {
                // this item's partial slot is its index among the prefill items
                float *pp = a.part + (((int64_t)wi * a.n_head_kv + hk) * M + n) * PART_STRIDE;
                pp[0] = m_run;
                pp[1] = l_run;
#pragma unroll
                for (int c = 0; c < 128; c += 4)
                    *reinterpret_cast<float4 *>(pp + 4 + c) = make_float4(ov[c], ov[c + 1], ov[c + 2], ov[c + 3]);
                __threadfence();
                tc::named_bar(1, 128);
                if (n == 0) {
                    const int32_t prev = atomicAdd(&a.p.counters[it.block * a.n_head_kv + hk], 1);
                    x.flag = (prev == it.nitems - 1) ? 1 : 0;
                }
                tc::named_bar(1, 128);
                if (x.flag) {
                    // merge.  Step 1: each thread reduces its own row's maxima and sums;
                    // step 2: four threads per row, 32 values each, all loads independent.
                    // The P buffer is free here and holds the per-row results.
                    __threadfence();
                    const int32_t first = a.p.blk_item0[it.block] - a.p.cap_dec;
                    const int64_t istride = (int64_t)a.n_head_kv * M * PART_STRIDE;
                    const float *base = a.part + ((int64_t)first * a.n_head_kv + hk) * M * PART_STRIDE;
                    float *mrow = reinterpret_cast<float *>(smem + OFF_P);
                    float *irow = mrow + M;
                    int32_t *rrow = reinterpret_cast<int32_t *>(irow + M);
                    {
                        const float *pr = base + (int64_t)n * PART_STRIDE;
                        float M_ = -INFINITY;
                        for (int32_t q = 0; q < it.nitems; ++q) M_ = fmaxf(M_, __ldcg(pr + q * istride));
                        float L = 0.f;
                        if (M_ != -INFINITY)
                            for (int32_t q = 0; q < it.nitems; ++q) {
                                const float mk = __ldcg(pr + q * istride);
                                if (mk != -INFINITY) L = fmaf(__ldcg(pr + q * istride + 1), ex2_approx(mk - M_), L);
                            }
                        mrow[n] = M_;
                        irow[n] = L > 0.f ? 1.f / L : 0.f;
                        rrow[n] = row;
                    }
                    tc::named_bar(1, 128);
                    const int32_t qd = n & 3;            // which 32 values of the row
#pragma unroll 1
                    for (int32_t pass = 0; pass < 4; ++pass) {
                        const int32_t r = pass * 32 + (n >> 2);
                        const int32_t orow_id = rrow[r];
                        const float Mr = mrow[r];
                        const float inv = irow[r];
                        float acc[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) acc[c] = 0.f;
                        if (orow_id >= 0 && Mr != -INFINITY) {
                            const float *pr = base + (int64_t)r * PART_STRIDE;
                            for (int32_t q = 0; q < it.nitems; ++q) {
                                const float *pq = pr + q * istride;
                                const float mk = __ldcg(pq);
                                float4 v[8];
#pragma unroll
                                for (int c = 0; c < 8; ++c)
                                    v[c] = __ldcg(reinterpret_cast<const float4 *>(pq + 4 + 32 * qd) + c);
                                const float sc = mk == -INFINITY ? 0.f : ex2_approx(mk - Mr);
#pragma unroll
                                for (int c = 0; c < 8; ++c) {
                                    acc[4 * c + 0] = fmaf(v[c].x, sc, acc[4 * c + 0]);
                                    acc[4 * c + 1] = fmaf(v[c].y, sc, acc[4 * c + 1]);
                                    acc[4 * c + 2] = fmaf(v[c].z, sc, acc[4 * c + 2]);
                                    acc[4 * c + 3] = fmaf(v[c].w, sc, acc[4 * c + 3]);
                                }
                            }
                        }
                        if (orow_id >= 0) {
                            float *dst = a.o + ((int64_t)orow_id * a.n_head + hk * G + (r % G)) * 128 + 32 * qd;
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                reinterpret_cast<float4 *>(dst)[c] = make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv,
                                                                                 acc[4 * c + 2] * inv, acc[4 * c + 3] * inv);
                        }
                    }
                    tc::named_bar(1, 128);   // the P buffer is written again by the next item
                    if (n == 0) a.p.counters[it.block * a.n_head_kv + hk] = 0;
                }
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (*fail && tid == 0) kvd::report(a.err, kvd::DERR_MMA_TIMEOUT);
    if (warp == 5) {
        tc::fence_after();
        tc::dealloc(tmem, TMEM_COLS);
    }
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
    return cudaGetLastError();
}

}  // namespace kvk
