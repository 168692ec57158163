// PoissonComp on the GPU: importance scores, water-filling, the Philox Poisson sample, compaction
// of H u S into device memory and the token-level key sketch.
// Paper: "Verify Before You Fetch: Reliable KV Cache Compression for LLM Inference",
// Algorithm 1 / Sec. 4.1 (eq. (3)) and Appendix A.1 (key sketch).
#include <algorithm>
#include <cmath>
#include <cstring>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "async.cuh"
#include "umma.cuh"

namespace cg = cooperative_groups;

namespace verkv {

namespace {

constexpr int kTauTok = 64;   // tokens per score tile
constexpr int kTauRows = 64;  // observation rows per chunk
constexpr int kTauLd = kHeadDim + 1;

// --------------------------------------------------------------------------------------------
// Importance scores (Algorithm 1, its scoring step), synthetic scorer: for the observation rows of the KV
// head's query-head group, p_j(i) = softmax_i(<Q_j, K_i>/sqrt(d)); tau_i = max_j p_j(i) / max.
// Pass 0 computes per (row, tile) the max logit and the sum of exp(logit - max); pass 1 turns the
// per-row totals into p and keeps the max over rows for each token.
// --------------------------------------------------------------------------------------------
template <typename T, int PASS>
__global__ void __launch_bounds__(256) tau_tile_kernel(const T* __restrict__ kv, int n, int R, int G, int W,
                                                       const float* __restrict__ obs_q, float scale,
                                                       float2* __restrict__ part, const float2* __restrict__ rowstat,
                                                       float* __restrict__ tau_raw, int* __restrict__ tau_max)
{
    extern __shared__ float smem[];
    float* Ks = smem;                        // [kTauTok][kTauLd]
    float* Qs = Ks + kTauTok * kTauLd;       // [kTauRows][kTauLd]
    float* Ls = Qs + kTauRows * kTauLd;      // [kTauRows][kTauTok + 1]
    float* best = Ls + kTauRows * (kTauTok + 1);  // [kTauTok]
    const int h = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x;
    const int t0 = tile * kTauTok;
    const int ntiles = gridDim.x;
    const int64_t head_base = (int64_t)h * n * 2 * kHeadDim;
    for (int e = tid; e < kTauTok * kHeadDim; e += blockDim.x) {
        int t = e / kHeadDim, c = e % kHeadDim;
        float v = 0.f;
        if (t0 + t < n) v = Elt<T>::load(kv, head_base + (int64_t)(t0 + t) * 2 * kHeadDim + c);
        Ks[t * kTauLd + c] = v;
    }
    if (PASS == 1 && tid < kTauTok) best[tid] = 0.f;
    const int tx = tid & 15, ty = tid >> 4;   // 16 x 16 threads, each a 4 x 4 block
    for (int r0 = 0; r0 < R; r0 += kTauRows) {
        __syncthreads();
        for (int e = tid; e < kTauRows * kHeadDim; e += blockDim.x) {
            int rr = e / kHeadDim, c = e % kHeadDim;
            int row = r0 + rr;
            float v = 0.f;
            if (row < R) {
                int g = row / W, w = row % W;
                v = obs_q[((int64_t)(h * G + g) * W + w) * kHeadDim + c];
            }
            Qs[rr * kTauLd + c] = v;
        }
        __syncthreads();
        float acc[4][4] = {};
        for (int c = 0; c < kHeadDim; ++c) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Qs[(ty + 16 * i) * kTauLd + c];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Ks[(tx + 16 * j) * kTauLd + c];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int rr = ty + 16 * i, t = tx + 16 * j;
                float l = acc[i][j] * scale;
                if (PASS == 1) {
                    int row = r0 + rr;
                    float p = 0.f;
                    if (row < R && t0 + t < n) {
                        float2 ms = rowstat[(int64_t)h * R + row];
                        p = __fdiv_rn(expf(l - ms.x), ms.y);
                    }
                    l = p;
                }
                Ls[rr * (kTauTok + 1) + t] = l;
            }
        __syncthreads();
        if (PASS == 0) {
            if (tid < kTauRows && r0 + tid < R) {
                float mx = -INFINITY;
                for (int t = 0; t < kTauTok && t0 + t < n; ++t) mx = fmaxf(mx, Ls[tid * (kTauTok + 1) + t]);
                float s = 0.f;
                for (int t = 0; t < kTauTok && t0 + t < n; ++t) s += expf(Ls[tid * (kTauTok + 1) + t] - mx);
                part[((int64_t)h * R + r0 + tid) * ntiles + tile] = make_float2(mx, s);
            }
        } else {
            if (tid < kTauTok) {
                float mx = best[tid];
                for (int rr = 0; rr < kTauRows; ++rr) mx = fmaxf(mx, Ls[rr * (kTauTok + 1) + tid]);
                best[tid] = mx;
            }
        }
    }
    if (PASS == 1) {
        __syncthreads();
        if (tid < kTauTok && t0 + tid < n) {
            tau_raw[(int64_t)h * n + t0 + tid] = best[tid];
            atomicMax(&tau_max[h], float_to_ordered(best[tid]));
        }
    }
}

// --------------------------------------------------------------------------------------------
// The same scores on the 5th-generation tensor cores, for bf16 keys and at most 128 observation rows
// per KV head: the logits of a tile of 128 tokens are one 128 x 128 x 128 product, A = the head's
// observation rows (fp32, split into three bf16 parts hi + mid + lo, which represent them to fp32
// precision; the products with the bf16 keys are exact and accumulate in fp32) and B = the tile's
// keys.  A stays in shared memory; key tiles arrive by cp.async into a two-stage ring in the
// 128-byte-swizzled K-major layout; one thread issues the 24 MMAs of a tile into one of two tensor-
// memory accumulators, so the next tile's MMAs overlap this tile's epilogue.  Epilogue: one thread
// per observation row.  Pass 0 keeps its row's running max and sum of exp(logit - max) over the
// block's tiles; pass 1 forms p = exp(logit - m) / Z and the max over rows of each token (a butterfly
// transpose-reduce per warp, then over the four lane quarters).  Sixteen warps: four per lane
// quarter of the accumulator, each on 32 of the tile's 128 columns.
// --------------------------------------------------------------------------------------------
constexpr int kTmmaN = 128;                       // tokens per tile
constexpr int kTmmaTileBytes = 128 * kHeadDim * 2;  // one bf16 operand tile (32 KiB)
constexpr int kTmmaStages = 3;                    // key tiles in flight
constexpr size_t kTmmaSmem = (size_t)(3 + kTmmaStages) * kTmmaTileBytes + 1024;   // A x 3, B ring, alignment slack

constexpr int kTmmaThreads = 512;   // 16 warps: 4 per tensor-memory lane quarter, 32 columns each

template <int PASS>
__global__ void __launch_bounds__(kTmmaThreads, 1) tau_mma_kernel(const __nv_bfloat16* __restrict__ kv, int n, int R,
                                                                  int G, int W, const float* __restrict__ obs_q,
                                                                  float scale, float2* __restrict__ part,
                                                                  const float2* __restrict__ rowstat,
                                                                  float* __restrict__ tau_raw, int* __restrict__ tau_max,
                                                                  int* __restrict__ err)
{
    extern __shared__ unsigned char dsm_raw[];
    __shared__ __align__(8) unsigned long long bar[2];
    __shared__ unsigned tbase;
    __shared__ float cmax[4][kTmmaN];        // pass 1: per lane quarter, max over its 32 rows of each column
    __shared__ float2 rpart[4][128];         // pass 0: per column group, each row's (max, sum)
    __shared__ float bred[kTmmaThreads / 32];
    // operand tiles must start on 1024-byte boundaries of the shared window
    unsigned char* dsm = dsm_raw + ((1024u - (umma_smem_u32(dsm_raw) & 1023u)) & 1023u);
    unsigned char* sA = dsm;                        // three 32 KiB parts of A
    unsigned char* sB = dsm + 3 * kTmmaTileBytes;   // kTmmaStages 32 KiB key stages
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quarter = warp & 3, cgrp = warp >> 2;   // lane quarter (rows 32 q ..) and column group (32 cg ..)
    const int row = 32 * quarter + lane;
    const int h = blockIdx.y;
    const int ntiles = (n + kTmmaN - 1) / kTmmaN;
    const int per = (ntiles + gridDim.x - 1) / gridDim.x;
    const int tb = min(ntiles, (int)blockIdx.x * per), nt = min(ntiles, tb + per) - tb;

    // A: the observation rows of the head's query-head group, split into bf16 hi + mid + lo
    for (int e = tid; e < 128 * kHeadDim; e += kTmmaThreads) {
        const int r = e / kHeadDim, k = e % kHeadDim;
        float v = 0.f;
        if (r < R) v = obs_q[((int64_t)(h * G + r / W) * W + r % W) * kHeadDim + k];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const float r1 = __fsub_rn(v, __bfloat162float(hi));
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(r1, __bfloat162float(mid)));
        const unsigned off = umma_sw128_offset(r, k, 128);
        *reinterpret_cast<__nv_bfloat16*>(sA + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sA + kTmmaTileBytes + off) = mid;
        *reinterpret_cast<__nv_bfloat16*>(sA + 2 * kTmmaTileBytes + off) = lo;
    }
    // keys of local tile i into stage i % kTmmaStages (one copy group per call, possibly empty)
    auto load_b = [&](int i) {
        if (i < nt) {
            const int tok0 = (tb + i) * kTmmaN;
            unsigned char* dst = sB + (i % kTmmaStages) * kTmmaTileBytes;
            for (int c = tid; c < kTmmaN * 16; c += kTmmaThreads) {
                const int r = c >> 4, cc = c & 15, tok = tok0 + r;
                const unsigned off = (unsigned)((cc >> 3) * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + (((cc & 7) ^ (r & 7)) << 4));
                if (tok < n) cp_async16(dst + off, kv + ((int64_t)h * n + tok) * 2 * kHeadDim + cc * 8);
                else *reinterpret_cast<uint4*>(dst + off) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_commit();
    };
    if (warp == 0) umma_alloc(&tbase, 256);
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int k = 0; k < kTmmaStages; ++k) load_b(k);
    fence_proxy_async_smem();   // A (generic stores) -> tensor core
    umma_fence_before();
    __syncthreads();
    umma_fence_after();
    const unsigned tmem = tbase;
    constexpr unsigned idesc = umma_idesc_bf16_f32(128, kTmmaN);
    auto issue = [&](int i) {   // thread 0
        const unsigned d = tmem + (unsigned)((i & 1) * kTmmaN);
        const unsigned ab = umma_smem_u32(sA), bb = umma_smem_u32(sB + (i % kTmmaStages) * kTmmaTileBytes);
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ++ks)
                umma_mma(d, umma_desc_sw128(ab + sp * kTmmaTileBytes + umma_kstep_offset(ks, 128)),
                          umma_desc_sw128(bb + umma_kstep_offset(ks, kTmmaN)), idesc, sp > 0 || ks > 0);
        umma_commit(&bar[i & 1]);
    };
    float m_run = -INFINITY, z_run = 0.f, best = 0.f;
    float msub = 0.f, zinv = 1.f;
    if (PASS == 1 && row < R) {
        const float2 ms = rowstat[(int64_t)h * R + row];
        msub = ms.x;
        zinv = __fdiv_rn(1.0f, ms.y);
    }
    bool bad = false;
    if (nt > 0) {
        cp_async_wait<kTmmaStages - 1>();
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            umma_fence_after();
            issue(0);
        }
    }
    for (int i = 0; i < nt; ++i) {
        if (i + 1 < nt) {
            cp_async_wait<kTmmaStages - 2>();   // groups of tiles <= i + 1 are done
            fence_proxy_async_smem();
            umma_fence_before();
            __syncthreads();   // tile i + 1 has landed; the epilogue of tile i - 1 is done with its accumulator
            if (tid == 0) {
                umma_fence_after();
                issue(i + 1);
            }
        }
        if (!mbar_wait(&bar[i & 1], (unsigned)((i >> 1) & 1), kWaitLimit)) bad = true;
        umma_fence_after();
        load_b(i + kTmmaStages);   // stage i % kTmmaStages is free once the MMAs of tile i are done
        const int col0 = 32 * cgrp, tok0 = (tb + i) * kTmmaN + col0;
        const unsigned acc = tmem + ((unsigned)(32 * quarter) << 16) + (unsigned)((i & 1) * kTmmaN + col0);
        float v[32];
        umma_ld16(acc, *reinterpret_cast<float(*)[16]>(v));
        umma_ld16(acc + 16, *reinterpret_cast<float(*)[16]>(v + 16));
        if (PASS == 0) {
            float cm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v[j] = (row < R && tok0 + j < n) ? __fmul_rn(v[j], scale) : -INFINITY;
                cm = fmaxf(cm, v[j]);
            }
            if (cm > -INFINITY) {
                const float mn = fmaxf(m_run, cm);
                float zs = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) zs += __expf(v[j] - mn);
                z_run = z_run * __expf(m_run - mn) + zs;
                m_run = mn;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const bool ok = row < R && tok0 + j < n;
                v[j] = ok ? __expf(__fmul_rn(v[j], scale) - msub) * zinv : 0.f;
            }
            // butterfly transpose-reduce: lane l ends with the max over the warp's 32 rows of column col0 + l
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const bool upper = (lane & o) != 0;
#pragma unroll
                for (int j = 0; j < o; ++j) {
                    const float send = upper ? v[j] : v[j + o];
                    const float keep = upper ? v[j + o] : v[j];
                    v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
                }
            }
            cmax[quarter][col0 + lane] = v[0];
            __syncthreads();
            if (tid < kTmmaN) {
                const float p = fmaxf(fmaxf(cmax[0][tid], cmax[1][tid]), fmaxf(cmax[2][tid], cmax[3][tid]));
                const int tok = (tb + i) * kTmmaN + tid;
                if (tok < n) {
                    tau_raw[(int64_t)h * n + tok] = p;
                    best = fmaxf(best, p);
                }
            }
            __syncthreads();   // cmax is rewritten by the next tile
        }
        umma_fence_before();
    }
    cp_async_wait<0>();
    if (PASS == 0) {
        rpart[cgrp][row] = make_float2(m_run, z_run);
        __syncthreads();
        if (tid < 128 && tid < R) {
            // combine the four column groups of the row
            float M = -INFINITY;
            for (int c = 0; c < 4; ++c) M = fmaxf(M, rpart[c][tid].x);
            float Z = 0.f;
            if (M > -INFINITY)
                for (int c = 0; c < 4; ++c)
                    if (rpart[c][tid].x > -INFINITY) Z += rpart[c][tid].y * __expf(rpart[c][tid].x - M);
            part[((int64_t)h * R + tid) * gridDim.x + blockIdx.x] = make_float2(M, Z);
        }
    } else {
        best = warp_max(best);
        if (lane == 0) bred[warp] = best;
    }
    if (bad) *(volatile int*)err = 1;
    __syncthreads();
    if (PASS == 1 && tid == 0) {
        float b = 0.f;
        for (int w = 0; w < kTmmaThreads / 32; ++w) b = fmaxf(b, bred[w]);
        atomicMax(&tau_max[h], float_to_ordered(b));
    }
    if (warp == 0) {
        umma_fence_after();
        umma_dealloc(tmem, 256);
    }
}

__global__ void tau_rowstat_kernel(const float2* __restrict__ part, int ntiles, float2* __restrict__ rowstat, int rows)
{
    const int row = blockIdx.x * blockDim.y + threadIdx.y;
    if (row >= rows) return;
    const float2* p = part + (int64_t)row * ntiles;
    float mx = -INFINITY;
    for (int t = threadIdx.x; t < ntiles; t += 32) mx = fmaxf(mx, p[t].x);
    mx = warp_max(mx);
    double s = 0.0;
    for (int t = threadIdx.x; t < ntiles; t += 32) s += (double)p[t].y * exp((double)p[t].x - (double)mx);
    s = warp_sum(s);
    if (threadIdx.x == 0) rowstat[row] = make_float2(mx, (float)s);
}

// tau := tau_raw / max (or the caller's scores), clamped to [2^-38, 1]; sink and local := 1.
__global__ void tau_finish_kernel(float* __restrict__ tau, const float* __restrict__ src, const int* __restrict__ tau_max,
                                  int n, int n_sink, int n_local)
{
    const int h = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = src[(int64_t)h * n + i];
    if (tau_max) v = __fdiv_rn(v, ordered_to_float(tau_max[h]));
    v = tau_clamp(v);
    if (i < n_sink || i >= n - n_local) v = 1.0f;
    tau[(int64_t)h * n + i] = v;
}

// --------------------------------------------------------------------------------------------
// Water-filling (Algorithm 1, its water-filling step; eq. (3)).  With U the tokens outside the sink/local
// windows and B' = eta n - |I|, the constant is c = (B' - t) / S where t tokens of U are capped
// (c tau >= 1) and S is the exact sum of the other scores.  For a threshold theta let
// psi(theta) = (B' - #{tau > theta}) theta - sum_{tau <= theta} tau; the capped set is
// {tau > theta*} for the largest data value theta* with psi(theta*) < 0, and {theta > 0 :
// psi(theta) < 0} is an interval, so a bisection over the fp32 bit patterns finds it.  Sums are
// exact: clamped scores are integers in units of 2^-61, accumulated in 2 x 64-bit words and
// rounded to double once.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t tau_fixed(float t)
{
    const uint32_t b = __float_as_uint(t);
    const uint64_t m = (b & 0x7fffffu) | 0x800000u;
    const int e = (int)((b >> 23) & 0xff) - 127;
    return m << (e + 38);
}

struct WfPass {
    int cnt_gt;
    double s_le;
    uint32_t max_le;  // largest bit pattern <= u (0 if none)
    uint32_t min_gt;  // smallest bit pattern > u (0xffffffff if none)
    bool below;       // psi(u) < 0: (B' - cnt_gt) u < s_le
};

// One bisection step, evaluated by the C CTAs of a head's cluster over their slices [i0, i1) of U:
// per CTA the warps' partials and the CTA's totals (in `tot[par]`, double-buffered by step parity),
// then every CTA combines all C totals through distributed shared memory.  The sums and extremes are
// integers, so every CTA obtains the same totals and takes the same bisection branch.
struct WfTot {
    unsigned long long lo, hi;
    int cnt;
    unsigned int max_le, min_gt, pad;
};

__device__ WfPass wf_pass(cg::cluster_group& cl, const float* __restrict__ t, int i0, int i1, uint32_t u,
                          double bprime, WfTot* wp, WfTot* tot, int par, WfPass* res)
{
    unsigned long long lo = 0, hi = 0;
    int cnt = 0;
    uint32_t mx = 0, mn = 0xffffffffu;
#pragma unroll 8
    for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
        const uint32_t b = __float_as_uint(t[i]);
        if (b > u) { ++cnt; mn = min(mn, b); }
        else {
            const uint64_t f = tau_fixed(t[i]);
            lo += f & 0xffffffffull;
            hi += f >> 32;
            mx = max(mx, b);
        }
    }
    lo = warp_sum(lo);
    hi = warp_sum(hi);
    cnt = warp_sum(cnt);
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) wp[warp] = WfTot{lo, hi, cnt, mx, mn, 0u};
    __syncthreads();
    if (warp == 0) {
        unsigned long long l2 = lane < nw ? wp[lane].lo : 0ull, h2 = lane < nw ? wp[lane].hi : 0ull;
        int c2 = lane < nw ? wp[lane].cnt : 0;
        unsigned int x2 = lane < nw ? wp[lane].max_le : 0u, n2 = lane < nw ? wp[lane].min_gt : 0xffffffffu;
        l2 = warp_sum(l2);
        h2 = warp_sum(h2);
        c2 = warp_sum(c2);
        for (int o = 16; o > 0; o >>= 1) {
            x2 = max(x2, __shfl_xor_sync(0xffffffffu, x2, o));
            n2 = min(n2, __shfl_xor_sync(0xffffffffu, n2, o));
        }
        if (lane == 0) tot[par] = WfTot{l2, h2, c2, x2, n2, 0u};
    }
    cl.sync();   // every CTA's totals of this step are in place (and the previous step's were read)
    // one thread combines them and does the double-precision part (fp64 is slow on this part), the
    // block reads the result
    if (threadIdx.x == 0) {
        unsigned long long L = 0, Hh = 0;
        int C = 0;
        uint32_t MX = 0, MN = 0xffffffffu;
        for (int q = 0; q < (int)cl.num_blocks(); ++q) {
            const WfTot x = cl.map_shared_rank(tot, q)[par];
            L += x.lo;
            Hh += x.hi;
            C += x.cnt;
            MX = max(MX, x.max_le);
            MN = min(MN, x.min_gt);
        }
        WfPass r;
        r.cnt_gt = C;
        const uint64_t low64 = (Hh << 32) + L;
        const uint64_t carry = low64 < L ? 1 : 0;
        const uint64_t high64 = (Hh >> 32) + carry;
        r.s_le = ldexp(u128_to_double_rn(high64, low64), -61);
        r.max_le = MX;
        r.min_gt = MN;
        r.below = (bprime - (double)C) * (double)__uint_as_float(u) < r.s_le;
        *res = r;
    }
    __syncthreads();
    return *res;
}

constexpr int kWfCluster = 8;                 // CTAs per head
constexpr int kWaterfillSmem = 200 * 1024;    // a CTA's slice of the scores kept on chip up to 51200 tokens

__global__ void __launch_bounds__(1024) waterfill_kernel(const float* __restrict__ tau, int n, int n_sink,
                                                         int n_local, double budget, double* __restrict__ c_out,
                                                         int* __restrict__ capped_out, int* __restrict__ neartie)
{
    __shared__ WfTot wp[32], tot[2];
    __shared__ WfPass res;
    extern __shared__ __align__(16) float wf_tau[];   // this CTA's slice of the scores, when the launch gave room
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank(), C = (int)cl.num_blocks();
    const int h = blockIdx.y;
    const float* t = tau + (int64_t)h * n;
    const int nf = n_sink + n_local;
    const double bprime = budget - (double)nf;
    const int nu = n - nf;
    if (bprime >= (double)nu) {   // the same in every CTA of the cluster: none of them synchronises
        if (rank == 0 && threadIdx.x == 0) { c_out[h] = INFINITY; capped_out[h] = nu; }
        return;
    }
    // this CTA's slice of U
    const int per = (nu + C - 1) / C;
    int i0 = n_sink + min(nu, rank * per), i1 = n_sink + min(nu, (rank + 1) * per);
    unsigned dyn_bytes;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
    if ((size_t)(i1 - i0) * sizeof(float) <= dyn_bytes) {
        // every bisection step reads the whole slice: read it from HBM once
        for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) wf_tau[i - i0] = t[i];
        __syncthreads();
        t = wf_tau;
        i1 -= i0;
        i0 = 0;
    }
    int par = 0;
    auto pass = [&](uint32_t u) {
        const WfPass p = wf_pass(cl, t, i0, i1, u, bprime, wp, tot, par, &res);
        par ^= 1;
        return p;
    };
    auto pred = [&](uint32_t u) -> bool { return pass(u).below; };
    uint32_t lo = 1u, hi = 0x3f800000u;
    uint32_t ustar;
    if (pred(hi)) ustar = hi;
    else {
        while (hi - lo > 1u) {
            const uint32_t mid = lo + (hi - lo) / 2u;
            if (pred(mid)) lo = mid; else hi = mid;
        }
        ustar = lo;
    }
    const WfPass p = pass(ustar);
    // The same decision at the data values themselves (the form of the rule that walks the
    // sorted scores): the capped/uncapped boundary must be accepted at max_le and rejected at min_gt.
    bool tie_hi = false;
    if (p.min_gt != 0xffffffffu) tie_hi = pass(p.min_gt).below;
    cl.sync();   // no CTA leaves while another may still read its totals
    if (rank == 0 && threadIdx.x == 0) {
        const double c = (bprime - (double)p.cnt_gt) / p.s_le;
        int tie = tie_hi ? 1 : 0;
        if (p.max_le != 0 && !((bprime - (double)p.cnt_gt) * (double)__uint_as_float(p.max_le) < p.s_le)) tie = 1;
        c_out[h] = c;
        capped_out[h] = p.cnt_gt;
        if (tie) atomicAdd(neartie, 1);
    }
}

// --------------------------------------------------------------------------------------------
// r_i = min(1, c tau_i) rounded to fp32 (H = {r = 1}); Z_i = [u_i < r_i] (Algorithm 1, its split and sampling steps).
// --------------------------------------------------------------------------------------------
__global__ void sample_kernel(const float* __restrict__ tau, const double* __restrict__ c, int n, int n_sink,
                              int n_local, uint64_t seed, int layer, int seq, float* __restrict__ r_out,
                              uint8_t* __restrict__ flags)
{
    const int h = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int64_t k = (int64_t)h * n + i;
    float r;
    if (i < n_sink || i >= n - n_local) r = 1.0f;
    else {
        const double ct = c[h] * (double)tau[k];
        r = ct < 1.0 ? __double2float_rn(ct) : 1.0f;
    }
    r_out[k] = r;
    uint8_t f;
    if (r == 1.0f) f = 2;
    else f = poisson_uniform(seed, (uint32_t)i, (uint32_t)h, (uint32_t)layer, (uint32_t)seq) < r ? 1 : 0;
    flags[k] = f;
}

// Ordered compaction of one KV head: L list (with r in L order), resident list (H u S), H list.
// lpos[token] is the L index for tokens of L and -(H index) - 1 for tokens of H.  A cluster of
// kCompactCluster CTAs per head: each counts the four classes over its run of tokens, takes the
// counts of the runs before it from the other CTAs' shared memory as its starting offsets, and then
// compacts its run in order.
constexpr int kCompactCluster = 8;
__global__ void __launch_bounds__(1024) compact_kernel(const uint8_t* __restrict__ flags, const float* __restrict__ r,
                                                       int n, int32_t* __restrict__ lpos, int32_t* __restrict__ ltok,
                                                       float* __restrict__ rl, int32_t* __restrict__ lslot,
                                                       float2* __restrict__ lq,
                                                       int32_t* __restrict__ rtok,
                                                       int32_t* __restrict__ hslot, int32_t* __restrict__ counts)
{
    __shared__ int scratch[32];
    __shared__ int cnt4[4];   // this CTA's run: |L|, |H u S|, |H|, |S|
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank(), C = (int)cl.num_blocks();
    const int h = blockIdx.y;
    const int64_t base = (int64_t)h * n;
    // this CTA's run of tokens, in whole blocks of blockDim.x
    const int per = (((n + C - 1) / C) + (int)blockDim.x - 1) / (int)blockDim.x * (int)blockDim.x;
    const int j0 = min(n, rank * per), j1 = min(n, j0 + per);
    {
        int cL = 0, cR = 0, cH = 0, cS = 0;
        for (int i = j0 + threadIdx.x; i < j1; i += blockDim.x) {
            const int f = flags[base + i];
            cL += (f == 0 || f == 1);
            cR += (f == 1 || f == 2);
            cH += (f == 2);
            cS += (f == 1);
        }
        cL = warp_sum(cL);
        cR = warp_sum(cR);
        cH = warp_sum(cH);
        cS = warp_sum(cS);
        if (threadIdx.x < 4) cnt4[threadIdx.x] = 0;
        __syncthreads();
        if ((threadIdx.x & 31) == 0) {
            atomicAdd(&cnt4[0], cL);
            atomicAdd(&cnt4[1], cR);
            atomicAdd(&cnt4[2], cH);
            atomicAdd(&cnt4[3], cS);
        }
    }
    cl.sync();   // every run's counts are in place
    int offL = 0, offR = 0, offH = 0, offS = 0;
    for (int q = 0; q < rank; ++q) {
        const int* c4 = cl.map_shared_rank(cnt4, q);
        offL += c4[0];
        offR += c4[1];
        offH += c4[2];
        offS += c4[3];
    }
    int totL = offL, totR = offR, totH = offH, totS = offS;
    if (rank == C - 1 && threadIdx.x == 0) {
        totL += cnt4[0];
        totR += cnt4[1];
        totH += cnt4[2];
        totS += cnt4[3];
    }
    cl.sync();   // every CTA has read the counts it needs (none is read after this)
    for (int t0 = j0; t0 < j1; t0 += blockDim.x) {
        const int i = t0 + threadIdx.x;
        const int f = i < j1 ? flags[base + i] : -1;
        const int isL = (f == 0 || f == 1), isR = (f == 1 || f == 2), isH = (f == 2), isS = (f == 1);
        int tot1, tot2;
        const int ex1 = block_exclusive_scan(isL | (isR << 16), scratch, &tot1);
        const int ex2 = block_exclusive_scan(isH | (isS << 16), scratch, &tot2);
        const int pL = ex1 & 0xffff, pR = ex1 >> 16, pH = ex2 & 0xffff;
        if (i < j1) {
            if (isL) {
                ltok[base + offL + pL] = i;
                rl[base + offL + pL] = r[base + i];
                lslot[base + offL + pL] = isS ? offR + pR : -1;
                {
                    const float rr = r[base + i], cr = __fsub_rn(1.0f, rr);
                    lq[base + offL + pL] = make_float2(__fdiv_rn(cr, rr), __fdiv_rn(rr, cr));
                }
                lpos[base + i] = offL + pL;
            } else {
                lpos[base + i] = -(offH + pH) - 1;
            }
            if (isR) rtok[base + offR + pR] = i;
            if (isH) hslot[base + offH + pH] = offR + pR;
        }
        offL += tot1 & 0xffff;
        offR += tot1 >> 16;
        offH += tot2 & 0xffff;
        offS += tot2 >> 16;
        __syncthreads();
    }
    if (rank == C - 1 && threadIdx.x == 0) {
        counts[h * 4 + 0] = totH;
        counts[h * 4 + 1] = totL;
        counts[h * 4 + 2] = totS;
        counts[h * 4 + 3] = totR;
    }
}

// Copy the K/V rows of H u S (ascending tokens) into the resident cache; one warp per row.
__global__ void gather_resident_kernel(const unsigned char* __restrict__ src, int n, size_t row_bytes,
                                       const int32_t* __restrict__ rtok, const int32_t* __restrict__ counts,
                                       const int64_t* __restrict__ res_off, unsigned char* __restrict__ dst)
{
    const int h = blockIdx.y;
    const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
    const int m = counts[h * 4 + 3];
    for (int s = blockIdx.x * warps + (threadIdx.x >> 5); s < m; s += gridDim.x * warps) {
        const int tok = rtok[(int64_t)h * n + s];
        const uint4* from = reinterpret_cast<const uint4*>(src + ((int64_t)h * n + tok) * row_bytes);
        uint4* to = reinterpret_cast<uint4*>(dst + (res_off[h] + s) * (int64_t)row_bytes);
        for (size_t v = lane; v < row_bytes / 16; v += 32) to[v] = from[v];
    }
}

// --------------------------------------------------------------------------------------------
// Int8 sketch: per token s = max|k| / 127 (fp32), code = rint(k / s) clamped to [-127, 127].
// One warp per token, 4 channels per lane.
// --------------------------------------------------------------------------------------------
template <typename T>
__global__ void sketch_int8_kernel(const T* __restrict__ kv, int n, int n_kv, int8_t* __restrict__ codes,
                                   float* __restrict__ scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t tok = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tok >= (int64_t)n * n_kv) return;
    const T* k = kv + tok * 2 * kHeadDim;  // [h][i] flattened: tok = h * n + i
    float v[4];
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[j] = Elt<T>::load(k, lane * 4 + j);
        mx = fmaxf(mx, fabsf(v[j]));
    }
    mx = warp_max(mx);
    const float s = __fdiv_rn(mx, 127.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int q = 0;
        if (s > 0.f) {
            float x = rintf(__fdiv_rn(v[j], s));
            x = fminf(fmaxf(x, -127.f), 127.f);
            q = (int)x;
        }
        packed |= ((uint32_t)(q & 0xff)) << (8 * j);
    }
    reinterpret_cast<uint32_t*>(codes + tok * kHeadDim)[lane] = packed;
    if (lane == 0) scale[tok] = s;
}

// 2-bit sketch, step 1: energy of each rotate-half pair (p, p + d/2), summed in float-float per
// block of tokens and in double across the blocks.
template <typename T>
__global__ void pair_energy_kernel(const T* __restrict__ kv, int n, int tokens_per_block, double* __restrict__ energy)
{
    const int h = blockIdx.y, c = threadIdx.x;  // blockDim.x == kHeadDim
    const int i0 = blockIdx.x * tokens_per_block;
    const int i1 = min(n, i0 + tokens_per_block);
    // float-float accumulation (fp64 arithmetic is slow on this part): x^2 is rounded to fp32 once
    // (exact for bf16 keys) and the running sum carries its rounding error, about 2^-44 relative
    ff e = {0.f, 0.f};
#pragma unroll 8
    for (int i = i0; i < i1; ++i) {
        const float x = Elt<T>::load(kv, ((int64_t)h * n + i) * 2 * kHeadDim + c);
        const ff t = two_sum(e.hi, __fmul_rn(x, x));
        e = fast_two_sum(t.hi, __fadd_rn(e.lo, t.lo));
    }
    atomicAdd(&energy[h * (kHeadDim / 2) + (c % (kHeadDim / 2))], (double)e.hi + (double)e.lo);
}

// Step 2: the d/8 pairs of largest energy (ties: lower pair index), ascending.
__global__ void select_pairs_kernel(const double* __restrict__ energy, int32_t* __restrict__ pairs)
{
    constexpr int P = kHeadDim / 2, K = kHeadDim / 8;
    __shared__ double e[P];
    __shared__ int chosen[P];
    const int h = blockIdx.x, p = threadIdx.x;  // blockDim.x == P
    e[p] = energy[h * P + p];
    __syncthreads();
    int rank = 0;
    for (int q = 0; q < P; ++q) rank += (e[q] > e[p]) || (e[q] == e[p] && q < p);
    chosen[p] = rank < K;
    __syncthreads();
    if (chosen[p]) {
        int pos = 0;
        for (int q = 0; q < p; ++q) pos += chosen[q];
        pairs[h * K + pos] = p;
    }
}

__device__ __forceinline__ uint64_t spread_bits(uint32_t x)
{
    uint64_t v = x;
    v = (v | (v << 16)) & 0x0000FFFF0000FFFFull;
    v = (v | (v << 8)) & 0x00FF00FF00FF00FFull;
    v = (v | (v << 4)) & 0x0F0F0F0F0F0F0F0Full;
    v = (v | (v << 2)) & 0x3333333333333333ull;
    v = (v | (v << 1)) & 0x5555555555555555ull;
    return v;
}

// Step 3: per (group of `group` tokens, kept channel) zero = fp16(min), scale = fp16((max-min)/3),
// code = rint((k - zero) / scale) clamped to [0, 3].  One block of kSk2Warps warps per group: warp w
// takes every kSk2Warps-th token of the group, lane = kept channel; the warps' minima and maxima are
// combined in shared memory (min and max are exact, so every warp obtains the same zero and scale).
constexpr int kSk2Warps = 4;
template <typename T>
__global__ void __launch_bounds__(32 * kSk2Warps) sketch_2bit_kernel(const T* __restrict__ kv, int n, int group,
                                                                     const int32_t* __restrict__ pairs,
                                                                     uint64_t* __restrict__ codes,
                                                                     __half* __restrict__ zero,
                                                                     __half* __restrict__ scl)
{
    constexpr int NP = kHeadDim / 8, KEPT = kHeadDim / 4;
    static_assert(KEPT == 32, "a lane per kept channel");
    __shared__ float smn[kSk2Warps][KEPT], smx[kSk2Warps][KEPT];
    const int h = blockIdx.y, g = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ch = lane < NP ? pairs[h * NP + lane] : pairs[h * NP + lane - NP] + kHeadDim / 2;
    const int i0 = g * group, i1 = min(n, i0 + group);
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll 8
    for (int i = i0 + warp; i < i1; i += kSk2Warps) {
        const float v = Elt<T>::load(kv, ((int64_t)h * n + i) * 2 * kHeadDim + ch);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    smn[warp][lane] = mn;
    smx[warp][lane] = mx;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kSk2Warps; ++w) {
        mn = fminf(mn, smn[w][lane]);
        mx = fmaxf(mx, smx[w][lane]);
    }
    const __half zh = __float2half_rn(mn);
    const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
    const int ngroups = (n + group - 1) / group;
    if (warp == 0) {
        zero[((int64_t)h * ngroups + g) * KEPT + lane] = zh;
        scl[((int64_t)h * ngroups + g) * KEPT + lane] = sh;
    }
    const float zf = __half2float(zh), sf = __half2float(sh);
#pragma unroll 8
    for (int i = i0 + warp; i < i1; i += kSk2Warps) {
        const float v = Elt<T>::load(kv, ((int64_t)h * n + i) * 2 * kHeadDim + ch);
        int code = 0;
        if (sf > 0.f) {
            float x = rintf(__fdiv_rn(__fsub_rn(v, zf), sf));
            x = fminf(fmaxf(x, 0.f), 3.f);
            code = (int)x;
        }
        const uint32_t b0 = __ballot_sync(0xffffffffu, code & 1);
        const uint32_t b1 = __ballot_sync(0xffffffffu, code >> 1);
        if (lane == 0) codes[(int64_t)h * n + i] = spread_bits(b0) | (spread_bits(b1) << 1);
    }
}

// Exact sketch: keep the keys themselves ([h][n][d]).
template <typename T>
__global__ void copy_keys_kernel(const T* __restrict__ kv, int64_t rows, T* __restrict__ out)
{
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= rows * kHeadDim) return;
    const int64_t row = e / kHeadDim, c = e % kHeadDim;
    out[e] = kv[row * 2 * kHeadDim + c];
}

template <typename T>
verkv_status run_scores(Ctx& ctx, Slot& s, const T* kv, int n, const float* obs_q, int W, const float* tau_in,
                        cudaStream_t st)
{
    const verkv_config& cfg = ctx.cfg;
    const int Hkv = cfg.n_kv_heads;
    dim3 g1((n + 255) / 256, Hkv);
    if (!obs_q) {
        tau_finish_kernel<<<g1, 256, 0, st>>>(s.tau, tau_in, nullptr, n, cfg.n_sink, cfg.n_local);
        VK_LAUNCHED("tau_finish");
        return VERKV_OK;
    }
    const int R = ctx.G * W;
    const int ntiles = (n + kTauTok - 1) / kTauTok;
    // scratch kept by the context (grown when a call needs more; the stream is idle here, the compress
    // having synchronised it on entry): per-tile partials, row statistics, raw scores, head maxima
    auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
    const size_t b_part = up(sizeof(float2) * (size_t)Hkv * R * ntiles), b_row = up(sizeof(float2) * (size_t)Hkv * R),
                 b_raw = up(sizeof(float) * (size_t)Hkv * n), b_max = up(sizeof(int) * Hkv);
    const size_t need = b_part + b_row + b_raw + b_max;
    if (need > ctx.tau_ws_cap) {
        if (ctx.tau_ws) VK_CUDA(cudaFree(ctx.tau_ws));
        ctx.tau_ws = nullptr;
        ctx.tau_ws_cap = 0;
        VK_CUDA(cudaMalloc(&ctx.tau_ws, need));
        ctx.tau_ws_cap = need;
    }
    unsigned char* ws = static_cast<unsigned char*>(ctx.tau_ws);
    float2* part = reinterpret_cast<float2*>(ws);
    float2* rowstat = reinterpret_cast<float2*>(ws + b_part);
    float* tau_raw = reinterpret_cast<float*>(ws + b_part + b_row);
    int* tau_max = reinterpret_cast<int*>(ws + b_part + b_row + b_raw);
    VK_CUDA(cudaMemsetAsync(tau_max, 0x80, sizeof(int) * Hkv, st));  // ordered(-huge)
    const size_t smem = sizeof(float) * ((size_t)kTauTok * kTauLd + (size_t)kTauRows * kTauLd +
                                         (size_t)kTauRows * (kTauTok + 1) + kTauTok);
    static bool attr_done[2] = {false, false};
    if (!attr_done[sizeof(T) == 4]) {
        VK_CUDA(cudaFuncSetAttribute(tau_tile_kernel<T, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        VK_CUDA(cudaFuncSetAttribute(tau_tile_kernel<T, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        attr_done[sizeof(T) == 4] = true;
    }
    const float scale = (float)(1.0 / std::sqrt((double)kHeadDim));
    dim3 br(32, 8);
    if (sizeof(T) == 2 && R <= 128) {
        // tensor cores: one block per SM, each over a run of 128-token tiles of one KV head
        static bool mma_attr = false;
        if (!mma_attr) {
            VK_CUDA(cudaFuncSetAttribute(tau_mma_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmmaSmem));
            VK_CUDA(cudaFuncSetAttribute(tau_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmmaSmem));
            mma_attr = true;
        }
        const int mtiles = (n + kTmmaN - 1) / kTmmaN;
        const int cph = std::max(1, std::min(mtiles, (ctx.num_sms + Hkv - 1) / Hkv));
        const dim3 gm(cph, Hkv);
        const __nv_bfloat16* kvb = reinterpret_cast<const __nv_bfloat16*>(kv);
        tau_mma_kernel<0><<<gm, kTmmaThreads, kTmmaSmem, st>>>(kvb, n, R, ctx.G, W, obs_q, scale, part, nullptr, nullptr, nullptr,
                                                      ctx.d_err);
        VK_LAUNCHED("tau_mma");
        tau_rowstat_kernel<<<(Hkv * R + 7) / 8, br, 0, st>>>(part, cph, rowstat, Hkv * R);
        VK_LAUNCHED("tau_rowstat");
        tau_mma_kernel<1><<<gm, kTmmaThreads, kTmmaSmem, st>>>(kvb, n, R, ctx.G, W, obs_q, scale, nullptr, rowstat, tau_raw,
                                                      tau_max, ctx.d_err);
        VK_LAUNCHED("tau_mma");
    } else {
        dim3 gt(ntiles, Hkv);
        tau_tile_kernel<T, 0><<<gt, 256, smem, st>>>(kv, n, R, ctx.G, W, obs_q, scale, part, nullptr, nullptr, nullptr);
        VK_LAUNCHED("tau_tile");
        tau_rowstat_kernel<<<(Hkv * R + 7) / 8, br, 0, st>>>(part, ntiles, rowstat, Hkv * R);
        VK_LAUNCHED("tau_rowstat");
        tau_tile_kernel<T, 1><<<gt, 256, smem, st>>>(kv, n, R, ctx.G, W, obs_q, scale, nullptr, rowstat, tau_raw, tau_max);
        VK_LAUNCHED("tau_tile");
    }
    tau_finish_kernel<<<g1, 256, 0, st>>>(s.tau, tau_raw, tau_max, n, cfg.n_sink, cfg.n_local);
    VK_LAUNCHED("tau_finish");
    return VERKV_OK;
}

template <typename T>
verkv_status run_sketch(Ctx& ctx, Slot& s, const T* kv, int n, cudaStream_t st)
{
    const verkv_config& cfg = ctx.cfg;
    const int Hkv = cfg.n_kv_heads;
    if (cfg.sketch == VERKV_SKETCH_INT8) {
        const int64_t toks = (int64_t)Hkv * n;
        sketch_int8_kernel<T><<<(unsigned)((toks + 7) / 8), 256, 0, st>>>(kv, n, Hkv, s.codes8, s.scale8);
        VK_LAUNCHED("sketch_int8");
    } else if (cfg.sketch == VERKV_SKETCH_2BIT) {
        VK_CUDA(cudaMemsetAsync(s.energy, 0, sizeof(double) * Hkv * (kHeadDim / 2), st));
        const int tpb = 256;
        pair_energy_kernel<T><<<dim3((n + tpb - 1) / tpb, Hkv), kHeadDim, 0, st>>>(kv, n, tpb, s.energy);
        VK_LAUNCHED("pair_energy");
        select_pairs_kernel<<<Hkv, kHeadDim / 2, 0, st>>>(s.energy, s.pairs);
        VK_LAUNCHED("select_pairs");
        const int ngroups = (n + cfg.sketch_group - 1) / cfg.sketch_group;
        sketch_2bit_kernel<T><<<dim3(ngroups, Hkv), 32 * kSk2Warps, 0, st>>>(kv, n, cfg.sketch_group, s.pairs,
                                                                             s.codes2, s.zero2, s.scale2);
        VK_LAUNCHED("sketch_2bit");
    } else {
        const int64_t rows = (int64_t)Hkv * n;
        copy_keys_kernel<T><<<(unsigned)((rows * kHeadDim + 255) / 256), 256, 0, st>>>(
            kv, rows, reinterpret_cast<T*>(s.kexact));
        VK_LAUNCHED("copy_keys");
    }
    return VERKV_OK;
}

}  // namespace

void free_slot(Slot& s)
{
    void* ptrs[] = {s.tau, s.r, s.flags, s.lpos, s.ltok, s.rl, s.lslot, s.lq, s.rtok, s.hslot, s.counts, s.c, s.capped, s.kvres,
                    s.res_off, s.codes8, s.scale8, s.codes2, s.zero2, s.scale2, s.pairs, s.energy, s.kexact,
                    s.stage_of, s.stage, s.stage_off, s.stage_cnt};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    s = Slot();
}

// Decode-time growth: n_new rows per KV head (src [Hkv][n_new][row], 16-byte words) go after the head's
// resident rows and the rows appended before them.
__global__ void append_rows_kernel(const uint4* __restrict__ src, int n_new, int words, const int64_t* __restrict__ res_off,
                                   const int32_t* __restrict__ counts, int n_tail, uint4* __restrict__ kvres)
{
    const int kv = blockIdx.y;
    const int64_t row0 = res_off[kv] + counts[kv * 4 + 3] + n_tail;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n_new * words; e += gridDim.x * blockDim.x) {
        const int j = e / words, w = e % words;
        kvres[(row0 + j) * words + w] = src[((int64_t)kv * n_new + j) * words + w];
    }
}

verkv_status append_rows(Ctx& ctx, Slot& s, int n_new, const void* src, cudaStream_t st)
{
    const int words = (int)(2 * kHeadDim * ctx.elt / 16);
    const int blocks = std::max(1, std::min(64, (n_new * words + 255) / 256));
    append_rows_kernel<<<dim3(blocks, ctx.cfg.n_kv_heads), 256, 0, st>>>(
        static_cast<const uint4*>(src), n_new, words, s.res_off, s.counts, s.n_tail, static_cast<uint4*>(s.kvres));
    VK_CUDA(cudaGetLastError());
    s.n_tail += n_new;
    return VERKV_OK;
}

verkv_status compress_slot(Ctx& ctx, Slot& s, int layer, int seq, int n, const void* kv_host, const void* kv_dev,
                           const float* obs_q, int W, const float* tau, cudaStream_t st)
{
    const verkv_config& cfg = ctx.cfg;
    const int Hkv = cfg.n_kv_heads;
    const size_t hn = (size_t)Hkv * n;
    VK_CUDA(cudaStreamSynchronize(st));
    // the per-token arrays are kept across calls while the context fits (head stride is always n)
    if (n > s.cap_n) {
        void* keep_res = s.kvres;
        int64_t* keep_off = s.res_off;
        const size_t keep_cap = s.cap_res;
        void* keep_stage = s.stage;
        const size_t keep_cap_stage = s.cap_stage;
        s.kvres = nullptr;
        s.res_off = nullptr;
        s.stage = nullptr;
        free_slot(s);
        s.kvres = keep_res;
        s.res_off = keep_off;
        s.cap_res = keep_cap;
        s.stage = keep_stage;
        s.cap_stage = keep_cap_stage;
        const size_t hc = (size_t)Hkv * n;
        VK_CUDA(cudaMalloc(&s.tau, sizeof(float) * hc));
        VK_CUDA(cudaMalloc(&s.r, sizeof(float) * hc));
        VK_CUDA(cudaMalloc(&s.flags, hc));
        VK_CUDA(cudaMalloc(&s.lpos, sizeof(int32_t) * hc));
        VK_CUDA(cudaMalloc(&s.ltok, sizeof(int32_t) * hc));
        VK_CUDA(cudaMalloc(&s.rl, sizeof(float) * hc));
        VK_CUDA(cudaMalloc(&s.lslot, sizeof(int32_t) * hc));
        VK_CUDA(cudaMalloc(&s.lq, sizeof(float2) * hc));
        VK_CUDA(cudaMalloc(&s.rtok, sizeof(int32_t) * hc));
        VK_CUDA(cudaMalloc(&s.hslot, sizeof(int32_t) * hc));
        VK_CUDA(cudaMalloc(&s.counts, sizeof(int32_t) * Hkv * 4));
        VK_CUDA(cudaMalloc(&s.c, sizeof(double) * Hkv));
        VK_CUDA(cudaMalloc(&s.capped, sizeof(int32_t) * (Hkv + 1)));
        VK_CUDA(cudaMalloc(&s.stage_of, sizeof(int32_t) * hc));
        VK_CUDA(cudaMalloc(&s.stage_off, sizeof(int64_t) * (Hkv + 1)));
        VK_CUDA(cudaMalloc(&s.stage_cnt, sizeof(int32_t) * Hkv));
        if (!s.res_off) VK_CUDA(cudaMalloc(&s.res_off, sizeof(int64_t) * (Hkv + 1)));
        if (cfg.sketch == VERKV_SKETCH_INT8) {
            VK_CUDA(cudaMalloc(&s.codes8, hc * kHeadDim));
            VK_CUDA(cudaMalloc(&s.scale8, sizeof(float) * hc));
        } else if (cfg.sketch == VERKV_SKETCH_2BIT) {
            const size_t ng = (size_t)(n + cfg.sketch_group - 1) / cfg.sketch_group;
            VK_CUDA(cudaMalloc(&s.codes2, sizeof(uint64_t) * hc));
            VK_CUDA(cudaMalloc(&s.zero2, sizeof(__half) * Hkv * ng * (kHeadDim / 4)));
            VK_CUDA(cudaMalloc(&s.scale2, sizeof(__half) * Hkv * ng * (kHeadDim / 4)));
            VK_CUDA(cudaMalloc(&s.pairs, sizeof(int32_t) * Hkv * (kHeadDim / 8)));
            VK_CUDA(cudaMalloc(&s.energy, sizeof(double) * Hkv * (kHeadDim / 2)));
        } else {
            VK_CUDA(cudaMalloc(&s.kexact, hc * kHeadDim * ctx.elt));
        }
        s.cap_n = n;
    }
    s.live = false;
    s.n = n;
    s.kv_host = kv_host;
    const void* kv = kv_dev ? kv_dev : kv_host;
    VK_TIMING_BEGIN();
    verkv_status rc;
    if (cfg.kv_dtype == VERKV_DTYPE_BF16)
        rc = run_scores<__nv_bfloat16>(ctx, s, (const __nv_bfloat16*)kv, n, obs_q, W, tau, st);
    else
        rc = run_scores<float>(ctx, s, (const float*)kv, n, obs_q, W, tau, st);
    if (rc != VERKV_OK) return rc;

    VK_CUDA(cudaMemsetAsync(s.capped + Hkv, 0, sizeof(int32_t), st));
    static bool wf_attr = false;
    if (!wf_attr) {
        VK_CUDA(cudaFuncSetAttribute(waterfill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWaterfillSmem));
        wf_attr = true;
    }
    {
        // one cluster of kWfCluster CTAs per KV head, each over a slice of the scores
        const size_t slice = (size_t)((n + kWfCluster - 1) / kWfCluster) * sizeof(float);
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(kWfCluster, Hkv);
        lc.blockDim = dim3(1024);
        lc.dynamicSmemBytes = slice <= (size_t)kWaterfillSmem ? slice : 0;
        lc.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kWfCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        VK_CUDA(cudaLaunchKernelEx(&lc, waterfill_kernel, (const float*)s.tau, n, cfg.n_sink, cfg.n_local,
                                   cfg.eta * (double)n, s.c, s.capped, s.capped + Hkv));
    }
    VK_LAUNCHED("waterfill");
    sample_kernel<<<dim3((n + 255) / 256, Hkv), 256, 0, st>>>(s.tau, s.c, n, cfg.n_sink, cfg.n_local, cfg.seed, layer,
                                                            seq, s.r, s.flags);
    VK_LAUNCHED("sample");
    {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(kCompactCluster, Hkv);
        lc.blockDim = dim3(1024);
        lc.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kCompactCluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        VK_CUDA(cudaLaunchKernelEx(&lc, compact_kernel, (const uint8_t*)s.flags, (const float*)s.r, n, s.lpos, s.ltok,
                                   s.rl, s.lslot, s.lq, s.rtok, s.hslot, s.counts));
    }
    VK_LAUNCHED("compact");

    std::vector<int32_t> counts((size_t)Hkv * 4), capped((size_t)Hkv + 1);
    std::vector<double> cval(Hkv);
    VK_CUDA(cudaMemcpyAsync(counts.data(), s.counts, sizeof(int32_t) * Hkv * 4, cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaMemcpyAsync(capped.data(), s.capped, sizeof(int32_t) * (Hkv + 1), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaMemcpyAsync(cval.data(), s.c, sizeof(double) * Hkv, cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    s.res_off_host.assign((size_t)Hkv + 1, 0);
    s.stats.assign((size_t)Hkv, verkv_head_stats{});
    // room for tokens appended at decode time after each head's resident rows (empty until then)
    s.n_tail = 0;
    s.cap_tail = std::max(0, std::min(ctx.append_rows, ctx.cfg.max_tokens - n));
    int max_res = 0;
    for (int h = 0; h < Hkv; ++h) {
        verkv_head_stats& hs = s.stats[h];
        hs.c = cval[h];
        hs.n_capped = capped[h];
        hs.n_h = counts[h * 4 + 0];
        hs.n_l = counts[h * 4 + 1];
        hs.n_s = counts[h * 4 + 2];
        hs.n_resident = counts[h * 4 + 3];
        s.res_off_host[h + 1] = s.res_off_host[h] + hs.n_resident + s.cap_tail;
        max_res = std::max(max_res, hs.n_resident);
    }
    const size_t row_bytes = 2 * kHeadDim * ctx.elt;
    const size_t need_res = std::max<size_t>(1, (size_t)s.res_off_host[Hkv]);
    if (need_res > s.cap_res) {
        if (s.kvres) VK_CUDA(cudaFree(s.kvres));
        s.kvres = nullptr;
        s.cap_res = need_res + need_res / 8;   // room for the next sample of the same size
        VK_CUDA(cudaMalloc(&s.kvres, s.cap_res * row_bytes));
    }
    VK_CUDA(cudaMemcpyAsync(s.res_off, s.res_off_host.data(), sizeof(int64_t) * (Hkv + 1), cudaMemcpyHostToDevice, st));
    // the staging cache starts empty: room for ceil(eta n) rows of L \ S per head by default (the size of
    // the resident sample again), every row of L \ S, or the set capacity
    s.stage_off_host.assign((size_t)Hkv + 1, 0);
    const int64_t eta_n = (int64_t)std::ceil(cfg.eta * (double)n);
    for (int h = 0; h < Hkv; ++h) {
        const int64_t fetchable = s.stats[h].n_l - s.stats[h].n_s;
        const int64_t want = ctx.stage_rows == VERKV_STAGE_ALL ? fetchable
                             : ctx.stage_rows == VERKV_STAGE_ETA_N ? eta_n : ctx.stage_rows;
        const int64_t cap = std::min<int64_t>(want, fetchable);
        s.stage_off_host[h + 1] = s.stage_off_host[h] + cap;
    }
    const size_t need_stage = (size_t)s.stage_off_host[Hkv];
    if (need_stage > s.cap_stage) {
        if (s.stage) VK_CUDA(cudaFree(s.stage));
        s.stage = nullptr;
        s.cap_stage = need_stage + need_stage / 8;
        VK_CUDA(cudaMalloc(&s.stage, s.cap_stage * row_bytes));
    }
    VK_CUDA(cudaMemcpyAsync(s.stage_off, s.stage_off_host.data(), sizeof(int64_t) * (Hkv + 1), cudaMemcpyHostToDevice,
                            st));
    VK_CUDA(cudaMemsetAsync(s.stage_of, 0xff, sizeof(int32_t) * hn, st));
    VK_CUDA(cudaMemsetAsync(s.stage_cnt, 0, sizeof(int32_t) * Hkv, st));
    if (max_res > 0) {
        gather_resident_kernel<<<dim3((max_res + 7) / 8, Hkv), 256, 0, st>>>(
            (const unsigned char*)kv, n, row_bytes, s.rtok, s.counts, s.res_off, (unsigned char*)s.kvres);
        VK_LAUNCHED("gather_resident");
    }
    if (cfg.kv_dtype == VERKV_DTYPE_BF16)
        rc = run_sketch<__nv_bfloat16>(ctx, s, (const __nv_bfloat16*)kv, n, st);
    else
        rc = run_sketch<float>(ctx, s, (const float*)kv, n, st);
    if (rc != VERKV_OK) return rc;
    VK_CUDA(cudaStreamSynchronize(st));
    s.live = true;
    return VERKV_OK;
}

}  // namespace verkv
