// K3a: GQA flash attention, decode path (memory bound).
//
// "llama.cpp and the ubatch", "The mask is doing the work" and "Chunked
// prefill is the same mechanism": o = softmax(q K^T / sqrt(d) + mask) V over
// the cells a row may see; masked cells contribute nothing.  "Iteration-Level
// Batching", "The budget that actually binds": the n_head / n_head_kv query
// heads of a group share one KV head.
//
// Design (sm_103a):
//  * grid = (CTA columns, KV heads); each CTA column owns an equal slice of
//    the concatenated visible-tile lists of all decode blocks (stream-K),
//    split at block boundaries into work items; a block is up to 16 query
//    vectors (rows sharing a first sequence id, times the GQA group), so every
//    K/V byte read serves all of them;
//  * warp 4 is the producer: it streams K and V tiles with TMA (2-D tensor
//    maps, 128-byte swizzle) into a 3-stage ring and, for tiles that are not
//    fully visible, the cells' visibility and positions into the same slot;
//    full/empty mbarriers, every wait bounded (a timeout sets the error word);
//  * warps 0-3 consume: scores with one thread per (cell, query parity), fp32
//    FMA on fp16 K; online softmax in base 2 with warp-shuffle max/sum; PV
//    with one thread per (d pair, cell parity);
//  * cells nobody in the block may see are never multiplied (masked scores
//    are replaced by -inf and PV skips such cells, so a NaN in an unused cell
//    cannot leak);
//  * the items of one block are merged by the last CTA to finish (atomic
//    counter, no spinning): O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.

#include "dev_common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace {

using kvi::TILE;
using kvi::DEC_QMAX;

constexpr int NCONS = 128;                      // consumer threads (warps 0-3)
constexpr int NT = NCONS + 32;                  // + producer warp
constexpr int STAGES = 3;
constexpr int BOX_BYTES = TILE * 128;           // 64 rows x 64 fp16
constexpr int STAGE_BYTES = 4 * BOX_BYTES;      // K lo, K hi, V lo, V hi
constexpr int PART_STRIDE = 132;                // m, l, pad, pad, o[128]
constexpr int HQ = DEC_QMAX / 2;
constexpr int PT_STRIDE = DEC_QMAX + 4;         // padded: 4-way instead of 16-way bank conflicts

struct Meta {                 // per stage: what the producer learned about the tile
    int32_t full;
    int32_t pad[3];
    int32_t cpos[TILE];
    uint8_t has[TILE];        // cell holds the block's sequence and is not from a later ubatch
};

struct __align__(16) Aux {
    Meta meta[STAGES];
    __half q[DEC_QMAX][128];      // queries as given (fp16)
    float s[DEC_QMAX][TILE];      // scores of the current tile (log2 units)
    float pt[TILE][PT_STRIDE];    // probabilities, cell-major
    float m[DEC_QMAX], l[DEC_QMAX], alpha[DEC_QMAX];
    int32_t rpos[DEC_QMAX];
    uint64_t full[STAGES], empty[STAGES];
    uint8_t anyvis[2][TILE];
    int32_t fail;
    int32_t flag;
};

constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + sizeof(Aux);

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

// Named barrier over the consumer warps that also ORs a predicate.
__device__ __forceinline__ bool cons_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r) : "r"((uint32_t)v), "r"(NCONS) : "memory");
    return r != 0;
}
__device__ __forceinline__ void cons_bar() { tc::named_bar(1, NCONS); }

__global__ void __launch_bounds__(NT, 2)
k_decode(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
         const kvk::DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *stages = smem;
    Aux &x = *reinterpret_cast<Aux *>(smem + (size_t)STAGES * STAGE_BYTES);
    volatile int32_t *fail = &x.fail;
    const int32_t tid = threadIdx.x;
    const int32_t lane = tid & 31, warp = tid >> 5;
    const int32_t hk = blockIdx.y;
    const int32_t G = a.gqa;
    const int32_t i0 = a.p.cta_item0[blockIdx.x];
    const int32_t i1 = a.p.cta_item0[blockIdx.x + 1];

    if ((kvd::smem_u32(smem) & 1023u) != 0) {   // TMA swizzle needs 1 KiB alignment
        if (tid == 0) kvd::report(a.err, kvd::DERR_BOUNDS);
        return;
    }
    if (tid == 0) {
        kvd::prefetch_tmap(&tm_k);
        kvd::prefetch_tmap(&tm_v);
        for (int s = 0; s < STAGES; ++s) {
            kvd::mbar_init(&x.full[s], 33);    // producer lane 0's expect_tx + 32 lanes
            kvd::mbar_init(&x.empty[s], 4);    // one arrival per consumer warp
        }
        x.fail = 0;
        kvd::fence_mbar_init();
    }
    __syncthreads();

    if (warp == 4) {
        // ======================= producer =======================
        int32_t k = 0;
        // wait outcomes and the loop condition are agreed by the whole warp, so a
        // failure never splits it in front of __syncwarp
        for (int32_t wi = i0; wi < i1 && __all_sync(0xffffffffu, *fail == 0); ++wi) {
            const kvk::WorkItem w = a.p.work[wi];
            const kvi::DevBlock b = a.u.blocks[w.block];
            const int32_t *list = a.p.tiles + (int64_t)w.block * a.p.tile_stride;
            const uint32_t *flg = a.p.flags + (int64_t)w.block * a.p.tile_stride;
            for (int32_t li = w.t0; li < w.t1; ++li) {
                const int32_t st = k % STAGES;
                if (k >= STAGES &&
                    !__all_sync(0xffffffffu, wait_or_fail(&x.empty[st], (uint32_t)((k / STAGES) - 1) & 1u, fail)))
                    break;
                const int32_t t = list[li];
                const bool full = (int32_t)(flg[t] & 0xffffu) == b.n_rows * TILE;
                if (lane == 0) {
                    uint8_t *sp = stages + (size_t)st * STAGE_BYTES;
                    const int32_t y = b.stream * a.u.kv_size + t * TILE;
                    const int32_t xk = hk * 128;
                    kvd::fence_proxy_async_smem();
                    kvd::mbar_arrive_expect_tx(&x.full[st], STAGE_BYTES);
                    kvd::tma_load_2d(sp, &tm_k, xk, y, &x.full[st]);
                    kvd::tma_load_2d(sp + BOX_BYTES, &tm_k, xk + 64, y, &x.full[st]);
                    kvd::tma_load_2d(sp + 2 * BOX_BYTES, &tm_v, xk, y, &x.full[st]);
                    kvd::tma_load_2d(sp + 3 * BOX_BYTES, &tm_v, xk + 64, y, &x.full[st]);
                    x.meta[st].full = full ? 1 : 0;
                }
                if (!full) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int32_t c = lane + 32 * r;
                        const int32_t j = t * TILE + c;
                        bool has = false;
                        int32_t cp = 0;
                        if (j < a.u.n_kv) {
                            const int64_t g = (int64_t)b.stream * a.u.kv_size + j;
                            const uint64_t wb = a.u.cell_bits[g * a.u.n_words + (b.seq0 >> 6)];
                            has = ((wb >> (b.seq0 & 63)) & 1ull) && a.u.cell_epoch[g] <= a.u.ub_epoch;
                            cp = a.u.cell_pos[g];
                        }
                        x.meta[st].has[c] = has ? 1 : 0;
                        x.meta[st].cpos[c] = cp;
                    }
                }
                __syncwarp();
                kvd::mbar_arrive(&x.full[st]);
                ++k;
            }
        }
        if (*fail && lane == 0) {
            // let copies already in flight land before the CTA's smem is released
            for (int32_t q = k > STAGES ? k - STAGES : 0; q < k; ++q)
                (void)kvd::mbar_wait_bounded(&x.full[q % STAGES], (uint32_t)(q / STAGES) & 1u);
        }
    } else {
        // ======================= consumers =======================
        int32_t k = 0;
        const int32_t c_cell = tid & (TILE - 1);   // scores: my cell
        const int32_t par = tid >> 6;              // scores: query parity / PV: cell parity
        const int32_t dp = (tid & 63) * 2;         // PV: my d pair
        bool failed = false;
        for (int32_t wi = i0; wi < i1 && !failed; ++wi) {
            const kvk::WorkItem w = a.p.work[wi];
            const kvi::DevBlock b = a.u.blocks[w.block];
            const int32_t NQ = b.n_rows * G;
            for (int32_t e = tid; e < NQ * 16; e += NCONS) {
                const int32_t n = e >> 4, dd = (e & 15) * 8;
                const int32_t row = a.u.perm[b.row0 + n / G];
                const int32_t h = hk * G + (n % G);
                *reinterpret_cast<uint4 *>(&x.q[n][dd]) = *reinterpret_cast<const uint4 *>(
                    a.q + ((int64_t)row * a.n_head + h) * 128 + dd);
            }
            if (tid < DEC_QMAX) {
                x.m[tid] = -INFINITY;
                x.l[tid] = 0.f;
                x.rpos[tid] = tid < b.n_rows ? a.u.rows[a.u.perm[b.row0 + tid]].pos : 0;
            }
            float acc[DEC_QMAX][2];
#pragma unroll
            for (int n = 0; n < DEC_QMAX; ++n) acc[n][0] = acc[n][1] = 0.f;
            cons_bar();

            for (int32_t li = w.t0; li < w.t1; ++li) {
                const int32_t st = k % STAGES;
                const bool ok = wait_or_fail(&x.full[st], (uint32_t)(k / STAGES) & 1u, fail);
                if (cons_bar_or(!ok)) { failed = true; break; }
                const uint8_t *sp = stages + (size_t)st * STAGE_BYTES;
                const int32_t vb = k & 1;
                // ---- phase A: visibility and scores ----
                const bool full = x.meta[st].full != 0;
                const bool has = full || x.meta[st].has[c_cell];
                const int32_t cpos = full ? 0 : x.meta[st].cpos[c_cell];
                float dot[HQ];
#pragma unroll
                for (int q = 0; q < HQ; ++q) dot[q] = 0.f;
                if (has) {
#pragma unroll 4
                    for (int ch = 0; ch < 16; ++ch) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(
                            sp + (ch >> 3) * BOX_BYTES + kvd::swz128(c_cell, ch & 7));
                        const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
                        float kf[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(h2[e]);
                            kf[2 * e] = f.x;
                            kf[2 * e + 1] = f.y;
                        }
#pragma unroll
                        for (int q = 0; q < HQ; ++q) {
                            const int n = 2 * q + par;
                            if (n < NQ) {
                                const uint4 qr = *reinterpret_cast<const uint4 *>(&x.q[n][ch * 8]);
                                const __half2 *q2 = reinterpret_cast<const __half2 *>(&qr);
                                float d0 = dot[q];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 qf = __half22float2(q2[e]);
                                    d0 = fmaf(qf.x, kf[2 * e], d0);
                                    d0 = fmaf(qf.y, kf[2 * e + 1], d0);
                                }
                                dot[q] = d0;
                            }
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < HQ; ++q) {
                    const int n = 2 * q + par;
                    if (n < NQ) {
                        const bool vis = has && (full || !a.u.causal || cpos <= x.rpos[n / G]);
                        x.s[n][c_cell] = vis ? dot[q] * a.scale_log2 : -INFINITY;
                    }
                }
                if (par == 0) {
                    const bool any = has && (full || !a.u.causal || cpos <= b.pos_max);
                    x.anyvis[vb][c_cell] = any ? 1 : 0;
                }
                cons_bar();
                // ---- phase B: online softmax, one warp per query (strided) ----
                for (int n = warp; n < NQ; n += NCONS / 32) {
                    const float s0 = x.s[n][lane], s1 = x.s[n][lane + 32];
                    float tmax = fmaxf(s0, s1);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                    const float m_old = x.m[n];
                    const float m_new = fmaxf(m_old, tmax);
                    float p0 = 0.f, p1 = 0.f, alpha = 1.f;
                    if (m_new != -INFINITY) {
                        p0 = exp2f(s0 - m_new);
                        p1 = exp2f(s1 - m_new);
                        alpha = exp2f(m_old - m_new);
                    }
                    float ls = p0 + p1;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
                    x.pt[lane][n] = p0;
                    x.pt[lane + 32][n] = p1;
                    if (lane == 0) {
                        x.m[n] = m_new;
                        x.l[n] = x.l[n] * alpha + ls;
                        x.alpha[n] = alpha;
                    }
                }
                cons_bar();
                // ---- phase C: O = alpha O + P V, cells of my parity ----
#pragma unroll
                for (int n = 0; n < DEC_QMAX; ++n) {
                    if (n < NQ) {
                        const float al = x.alpha[n];
                        acc[n][0] *= al;
                        acc[n][1] *= al;
                    }
                }
                const int ch = dp >> 3;
                const uint32_t vin = (uint32_t)(dp & 7) * 2u;
                const uint8_t *vbase = sp + 2 * BOX_BYTES + (ch >> 3) * BOX_BYTES;
                for (int c = par; c < TILE; c += 2) {
                    if (!x.anyvis[vb][c]) continue;
                    const float2 v = __half22float2(
                        *reinterpret_cast<const __half2 *>(vbase + kvd::swz128(c, ch & 7) + vin));
#pragma unroll
                    for (int n4 = 0; n4 < DEC_QMAX; n4 += 4) {
                        if (n4 < NQ) {
                            const float4 p = *reinterpret_cast<const float4 *>(&x.pt[c][n4]);
                            acc[n4 + 0][0] = fmaf(p.x, v.x, acc[n4 + 0][0]);
                            acc[n4 + 0][1] = fmaf(p.x, v.y, acc[n4 + 0][1]);
                            acc[n4 + 1][0] = fmaf(p.y, v.x, acc[n4 + 1][0]);
                            acc[n4 + 1][1] = fmaf(p.y, v.y, acc[n4 + 1][1]);
                            acc[n4 + 2][0] = fmaf(p.z, v.x, acc[n4 + 2][0]);
                            acc[n4 + 2][1] = fmaf(p.z, v.y, acc[n4 + 2][1]);
                            acc[n4 + 3][0] = fmaf(p.w, v.x, acc[n4 + 3][0]);
                            acc[n4 + 3][1] = fmaf(p.w, v.y, acc[n4 + 3][1]);
                        }
                    }
                }
                // release the stage (K, V and its metadata)
                __syncwarp();
                if (lane == 0) kvd::mbar_arrive(&x.empty[st]);
                ++k;
            }
            if (failed) break;

            // ---- merge the two cell parities (s and pt hold 16 x 128 floats) ----
            cons_bar();
            float *red = &x.s[0][0];
            if (par == 1) {
#pragma unroll
                for (int n = 0; n < DEC_QMAX; ++n) {
                    if (n < NQ) {
                        red[n * 128 + dp] = acc[n][0];
                        red[n * 128 + dp + 1] = acc[n][1];
                    }
                }
            }
            cons_bar();
            const int32_t nitems = a.p.blk_nitems[w.block];
            if (par == 0) {
#pragma unroll
                for (int n = 0; n < DEC_QMAX; ++n) {
                    if (n < NQ) {
                        acc[n][0] += red[n * 128 + dp];
                        acc[n][1] += red[n * 128 + dp + 1];
                    }
                }
                if (nitems == 1) {
#pragma unroll
                    for (int n = 0; n < DEC_QMAX; ++n) {
                        if (n < NQ) {
                            const float l = x.l[n];
                            const float inv = l > 0.f ? 1.f / l : 0.f;
                            const int32_t row = a.u.perm[b.row0 + n / G];
                            const int32_t h = hk * G + (n % G);
                            *reinterpret_cast<float2 *>(a.o + ((int64_t)row * a.n_head + h) * 128 + dp) =
                                make_float2(acc[n][0] * inv, acc[n][1] * inv);
                        }
                    }
                } else {
                    float *pp = a.part + ((int64_t)wi * a.n_head_kv + hk) * DEC_QMAX * PART_STRIDE;
#pragma unroll
                    for (int n = 0; n < DEC_QMAX; ++n) {
                        if (n < NQ) {
                            *reinterpret_cast<float2 *>(pp + n * PART_STRIDE + 4 + dp) = make_float2(acc[n][0], acc[n][1]);
                            if (dp == 0) {
                                pp[n * PART_STRIDE + 0] = x.m[n];
                                pp[n * PART_STRIDE + 1] = x.l[n];
                            }
                        }
                    }
                }
            }
            if (nitems > 1) {
                __threadfence();
                cons_bar();
                if (tid == 0) {
                    const int32_t prev = atomicAdd(&a.p.counters[w.block * a.n_head_kv + hk], 1);
                    x.flag = (prev == nitems - 1) ? 1 : 0;
                }
                cons_bar();
                if (x.flag) {
                    __threadfence();
                    const int32_t it0 = a.p.blk_item0[w.block];
                    for (int32_t e = tid; e < NQ * 64; e += NCONS) {
                        const int32_t n = e >> 6, d2 = (e & 63) * 2;
                        float M = -INFINITY;
                        for (int32_t q = 0; q < nitems; ++q) {
                            const float *pk = a.part + ((int64_t)(it0 + q) * a.n_head_kv + hk) * DEC_QMAX * PART_STRIDE
                                              + n * PART_STRIDE;
                            M = fmaxf(M, __ldcg(pk));
                        }
                        float L = 0.f, o0 = 0.f, o1 = 0.f;
                        if (M != -INFINITY) {
                            for (int32_t q = 0; q < nitems; ++q) {
                                const float *pk = a.part + ((int64_t)(it0 + q) * a.n_head_kv + hk) * DEC_QMAX * PART_STRIDE
                                                  + n * PART_STRIDE;
                                const float mk = __ldcg(pk);
                                if (mk == -INFINITY) continue;
                                const float sc = exp2f(mk - M);
                                L = fmaf(__ldcg(pk + 1), sc, L);
                                const float2 ov = __ldcg(reinterpret_cast<const float2 *>(pk + 4 + d2));
                                o0 = fmaf(ov.x, sc, o0);
                                o1 = fmaf(ov.y, sc, o1);
                            }
                        }
                        const float inv = L > 0.f ? 1.f / L : 0.f;
                        const int32_t row = a.u.perm[b.row0 + n / G];
                        const int32_t h = hk * G + (n % G);
                        *reinterpret_cast<float2 *>(a.o + ((int64_t)row * a.n_head + h) * 128 + d2) =
                            make_float2(o0 * inv, o1 * inv);
                    }
                    if (tid == 0) a.p.counters[w.block * a.n_head_kv + hk] = 0;
                }
            }
            cons_bar();
        }
    }
    __syncthreads();
    if (*fail && tid == 0) kvd::report(a.err, kvd::DERR_TMA_TIMEOUT);
}

}  // namespace

namespace kvk {

int32_t decode_ctas_per_sm() { return 2; }

cudaError_t launch_decode(const CUtensorMap *tm_k, const CUtensorMap *tm_v, const DecodeArgs &a,
                          int32_t grid_x, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    k_decode<<<dim3(grid_x, a.n_head_kv), NT, SMEM_BYTES, st>>>(*tm_k, *tm_v, a);
    return cudaGetLastError();
}

}  // namespace kvk
