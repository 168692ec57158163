// KVFetch on the GPU: sketch scores, the bounded-shrinkage fixed point, the Bernstein
// certificate, gains, ranking, k*, the union fetch from pinned host memory and the weighted
// attention.  Paper: "Verify Before You Fetch: Reliable KV Cache Compression for LLM Inference",
// Algorithm 2 / Sec. 4.2 (Definition 2 / eq. (5), Lemma 1 / eq. (7), eqs. (9)-(10), Theorem 2),
// Appendix A.1 (sketch), Appendix A.3.2 (decide / fetch / attention kernels: prior art).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace verkv {

namespace {

constexpr int kMaxBatch = 32;
constexpr int kTile = 128;      // token positions per score block (= 2-bit sketch group)
constexpr int kSelWidth = 4096; // candidates ranked on chip per row

struct Views {
    SlotView v[kMaxBatch];
};

struct DecodeArgs {
    int Hkv, Hq, G, ws_n, ws_npow2, gen, nsplit;
    float eps_f;
    double eps, ldelta;
    float inv_sqrt_d_f;
    ff inv_sqrt_d;
};

__device__ __forceinline__ int row_of(int b, int hq, int Hq) { return b * Hq + hq; }

// --------------------------------------------------------------------------------------------
// Per-row state init.
// --------------------------------------------------------------------------------------------
__global__ void init_rows_kernel(RowState* __restrict__ rows, Views views, DecodeArgs a, int B)
{
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= B * a.Hq) return;
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    RowState s;
    memset(&s, 0, sizeof(s));
    s.m_ord = float_to_ordered(-INFINITY);
    s.n_h = views.v[b].counts[kv * 4 + 0];
    s.n_l = views.v[b].counts[kv * 4 + 1];
    s.b_arg = -1;
    rows[row] = s;
}

// --------------------------------------------------------------------------------------------
// D1: sketch logits <q, k^_i>/sqrt(d) of the tokens of L, as float-float.  One thread per token
// position, all G query heads of the KV head.  The query side is split so that the bulk of each
// dot product is an exact fp32 sum of integer multiples of a power of two:
//   int8:  q = h1 + h2 + l2 with h1 on the grid 2^(E-8) and h2 on 2^(E-17) (|q| < 2^E); with
//          codes |c| <= 127 every partial sum of h1*c (and of h2*c) is an integer < 2^24 in
//          grid units, so it is exact; only the tiny l2 part rounds.
//   2-bit: kappa_j = q_j * scale_gj (exact two-product), split on the grid 2^(E-17) of the group;
//          codes are 0..3 and 32 channels, so the grid part is exact as well.
// --------------------------------------------------------------------------------------------
template <int G>
struct QSplitInt8 {
    float h1[G][kHeadDim], h2[G][kHeadDim], l2[G][kHeadDim];
};

template <int G>
__device__ void split_q_int8(const float* __restrict__ q, QSplitInt8<G>& s, float* red)
{
    // blockDim.x == kTile == kHeadDim: thread c owns channel c of every head
    const int c = threadIdx.x;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float v = q[g * kHeadDim + c];
        const float mx = block_max(fabsf(v), red);
        int E;
        frexpf(mx, &E);  // mx < 2^E
        const float h1 = ldexpf(rintf(ldexpf(v, 8 - E)), E - 8);
        const float l1 = __fsub_rn(v, h1);
        const float h2 = ldexpf(rintf(ldexpf(l1, 17 - E)), E - 17);
        s.h1[g][c] = h1;
        s.h2[g][c] = h2;
        s.l2[g][c] = __fsub_rn(l1, h2);
    }
}

__device__ __forceinline__ ff combine3(float s1, float s2, float s3)
{
    ff t = two_sum(s1, s2);
    return fast_two_sum(t.hi, __fadd_rn(t.lo, s3));
}

template <int G>
__global__ void __launch_bounds__(kTile) score_int8_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                           RowState* __restrict__ rows, float2* __restrict__ tl)
{
    __shared__ QSplitInt8<G> qs;
    __shared__ float red[32];
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int i = blockIdx.x * kTile + threadIdx.x;
    split_q_int8<G>(q + ((int64_t)b * a.Hq + kv * G) * kHeadDim, qs, red);
    __syncthreads();
    const int64_t hi_ = (int64_t)kv * n + i;
    const bool live = i < n && V.flags[hi_] != 2;
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    if (live) {
        float s1[G], s2[G], s3[G];
#pragma unroll
        for (int g = 0; g < G; ++g) s1[g] = s2[g] = s3[g] = 0.f;
        const uint4* crow = reinterpret_cast<const uint4*>(V.codes8 + hi_ * kHeadDim);
#pragma unroll 1
        for (int c16 = 0; c16 < kHeadDim / 16; ++c16) {
            const uint4 w4 = crow[c16];
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int bte = 0; bte < 4; ++bte) {
                    const int c = c16 * 16 + k * 4 + bte;
                    const float cf = (float)(int8_t)((w[k] >> (8 * bte)) & 0xff);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        s1[g] = __fmaf_rn(qs.h1[g][c], cf, s1[g]);
                        s2[g] = __fmaf_rn(qs.h2[g][c], cf, s2[g]);
                        s3[g] = __fmaf_rn(qs.l2[g][c], cf, s3[g]);
                    }
                }
            }
        }
        const float sc = V.scale8[hi_];
        const int li = V.lpos[hi_];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ff t = combine3(s1[g], s2[g], s3[g]);
            t = ff_mul(ff_mul_f(t, sc), a.inv_sqrt_d);
            const int row = row_of(b, kv * G + g, a.Hq);
            tl[(int64_t)row * a.ws_n + li] = make_float2(t.hi, t.lo);
            mloc[g] = t.hi;
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m = block_max(mloc[g], red);
        if (threadIdx.x == 0 && m > -INFINITY) atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_ord, float_to_ordered(m));
    }
}

template <int G>
__global__ void __launch_bounds__(kTile) score_2bit_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                           RowState* __restrict__ rows, float2* __restrict__ tl)
{
    constexpr int NP = kHeadDim / 8, KEPT = kHeadDim / 4;
    __shared__ float k1[G][KEPT], rho[G][KEPT];
    __shared__ ff zsum[G];
    __shared__ float red[32];
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int grp = blockIdx.x;  // kTile == sketch group
    const int ngroups = (n + kTile - 1) / kTile;
    if (grp >= ngroups) return;  // a shorter sequence of the batch
    const float* qb = q + ((int64_t)b * a.Hq + kv * G) * kHeadDim;
    // per (head, group): kappa_j = q_ch * scale, Z = sum_j q_ch * zero, split of kappa
    for (int gg = threadIdx.x >> 5; gg < G; gg += blockDim.x >> 5) {
        const int j = threadIdx.x & 31;
        const int p = V.pairs[kv * NP + (j % NP)];
        const int ch = j < NP ? p : p + kHeadDim / 2;
        const float qc = qb[gg * kHeadDim + ch];
        const int64_t pi = ((int64_t)kv * ngroups + grp) * KEPT + j;
        const float z = __half2float(V.zero2[pi]), sc = __half2float(V.scale2[pi]);
        const ff kap = two_prod(qc, sc);
        ff zz = two_prod(qc, z);
        zz = warp_sum_ff(zz);
        float mx = warp_max(fabsf(kap.hi));
        int E;
        frexpf(mx, &E);
        const float K1 = ldexpf(rintf(ldexpf(kap.hi, 17 - E)), E - 17);
        k1[gg][j] = K1;
        rho[gg][j] = __fadd_rn(__fsub_rn(kap.hi, K1), kap.lo);
        if (j == 0) zsum[gg] = zz;
    }
    __syncthreads();
    const int i = grp * kTile + threadIdx.x;
    const int64_t hi_ = (int64_t)kv * n + i;
    const bool live = i < n && V.flags[hi_] != 2;
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    if (live) {
        const uint64_t w = V.codes2[hi_];
        float s1[G], s2[G];
#pragma unroll
        for (int g = 0; g < G; ++g) s1[g] = s2[g] = 0.f;
#pragma unroll
        for (int j = 0; j < KEPT; ++j) {
            const float cf = (float)((w >> (2 * j)) & 3u);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                s1[g] = __fmaf_rn(k1[g][j], cf, s1[g]);
                s2[g] = __fmaf_rn(rho[g][j], cf, s2[g]);
            }
        }
        const int li = V.lpos[hi_];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            ff t = ff_add(zsum[g], two_sum(s1[g], s2[g]));
            t = ff_mul(t, a.inv_sqrt_d);
            const int row = row_of(b, kv * G + g, a.Hq);
            tl[(int64_t)row * a.ws_n + li] = make_float2(t.hi, t.lo);
            mloc[g] = t.hi;
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m = block_max(mloc[g], red);
        if (threadIdx.x == 0 && m > -INFINITY) atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_ord, float_to_ordered(m));
    }
}

// Exact float-float dot product <q, k>/sqrt(d) of one key row (fp32 or bf16 elements).
template <typename T>
__device__ __forceinline__ ff exact_logit(const float* __restrict__ q, const T* __restrict__ k, ff inv_sqrt_d)
{
    ff acc = {0.f, 0.f};
    float lo = 0.f;
#pragma unroll 8
    for (int c = 0; c < kHeadDim; ++c) {
        const ff p = two_prod(q[c], Elt<T>::load(k, c));
        const ff s = two_sum(acc.hi, p.hi);
        acc.hi = s.hi;
        lo = __fadd_rn(lo, __fadd_rn(s.lo, p.lo));
    }
    acc = fast_two_sum(acc.hi, lo);
    return ff_mul(acc, inv_sqrt_d);
}

// Exact sketch: the L logits from the keys themselves.
template <typename T, int G>
__global__ void __launch_bounds__(kTile) score_exact_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                            RowState* __restrict__ rows, float2* __restrict__ tl)
{
    __shared__ float qs[G][kHeadDim];
    __shared__ float red[32];
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    for (int e = threadIdx.x; e < G * kHeadDim; e += blockDim.x)
        qs[e / kHeadDim][e % kHeadDim] = q[((int64_t)b * a.Hq + kv * G) * kHeadDim + e];
    __syncthreads();
    const int i = blockIdx.x * kTile + threadIdx.x;
    const int64_t hi_ = (int64_t)kv * n + i;
    const bool live = i < n && V.flags[hi_] != 2;
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    if (live) {
        const T* k = reinterpret_cast<const T*>(V.kexact) + hi_ * kHeadDim;
        const int li = V.lpos[hi_];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const ff t = exact_logit<T>(qs[g], k, a.inv_sqrt_d);
            const int row = row_of(b, kv * G + g, a.Hq);
            tl[(int64_t)row * a.ws_n + li] = make_float2(t.hi, t.lo);
            mloc[g] = t.hi;
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m = block_max(mloc[g], red);
        if (threadIdx.x == 0 && m > -INFINITY) atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_ord, float_to_ordered(m));
    }
}

// Exact logits of the tokens of H (resident keys), by H index.
template <typename T, int G>
__global__ void __launch_bounds__(kTile) score_h_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                        RowState* __restrict__ rows, float2* __restrict__ th)
{
    __shared__ float qs[G][kHeadDim];
    __shared__ float red[32];
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int nh = V.counts[kv * 4 + 0];
    if (blockIdx.x * kTile >= nh) return;
    for (int e = threadIdx.x; e < G * kHeadDim; e += blockDim.x)
        qs[e / kHeadDim][e % kHeadDim] = q[((int64_t)b * a.Hq + kv * G) * kHeadDim + e];
    __syncthreads();
    const int k = blockIdx.x * kTile + threadIdx.x;
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    if (k < nh) {
        const int slot = V.hslot[(int64_t)kv * n + k];
        const T* key = reinterpret_cast<const T*>(V.kvres) + (V.res_off[kv] + slot) * 2 * kHeadDim;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const ff t = exact_logit<T>(qs[g], key, a.inv_sqrt_d);
            const int row = row_of(b, kv * G + g, a.Hq);
            th[(int64_t)row * a.ws_n + k] = make_float2(t.hi, t.lo);
            mloc[g] = t.hi;
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m = block_max(mloc[g], red);
        if (threadIdx.x == 0 && m > -INFINITY) atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_ord, float_to_ordered(m));
    }
}

// --------------------------------------------------------------------------------------------
// D2: weights w^_i = exp(t^_i - m) on L, w_i = exp(t_i - m) on H; D = sum_H w + sum_L w^ and
// sum_L w^ (1 - r) (the top of the beta bracket), float-float per thread.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ float weight_of(float2 t, float m)
{
    ff x = two_sum(t.x, -m);
    x = fast_two_sum(x.hi, __fadd_rn(x.lo, t.y));
    return ff_exp(x);
}

__global__ void __launch_bounds__(256) weights_kernel(Views views, DecodeArgs a, RowState* __restrict__ rows,
                                                      const float2* __restrict__ tl, const float2* __restrict__ th,
                                                      float* __restrict__ wl)
{
    __shared__ ff red[32];
    const int row = blockIdx.y;
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    const SlotView& V = views.v[b];
    RowState& R = rows[row];
    const int nl = R.n_l, nh = R.n_h;
    if (blockIdx.x * blockDim.x >= max(nl, nh)) return;
    const float m = ordered_to_float(R.m_ord);
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    ff d = {0.f, 0.f}, al = {0.f, 0.f};
    if (j < nl) {
        const float w = weight_of(tl[(int64_t)row * a.ws_n + j], m);
        wl[(int64_t)row * a.ws_n + j] = w;
        const float r = V.rl[(int64_t)kv * V.n + j];
        d = ff_add_f(d, w);
        al = two_prod(w, __fsub_rn(1.0f, r));
    }
    if (j < nh) d = ff_add_f(d, weight_of(th[(int64_t)row * a.ws_n + j], m));
    d = block_sum_ff(d, red);
    al = block_sum_ff(al, red);
    if (threadIdx.x == 0) {
        atomicAdd(&R.D, ff_to_double(d));
        atomicAdd(&R.alpha_sum, ff_to_double(al));
    }
}

// --------------------------------------------------------------------------------------------
// D3: the fixed point of Definition 2.  lambda_i(beta) = clip_[r,1](beta r / (w (1 - r))), so on
// the tokens with beta <= alpha_i = w_i (1 - r_i) lambda = r (bias alpha_i), with beta >= alpha_i /
// r_i lambda = 1 (no bias), and in between the bias is w_i - beta r_i / (1 - r_i).  The equation
// beta = sum_L w (1 - lambda(beta)) is G(beta) = beta (1 + R) - A - W = 0 with A, W, R sums over
// those classes; Newton's step on this piecewise-linear, increasing G is beta' = (A + W)/(1 + R)
// (exact once the classes are right), safeguarded by bisection on the bracket [lo, hi].
// Then lambda, a_i, v_i, b_i, eq. (7) and the no-fetch test (Algorithm 2, lines 2-5).
// --------------------------------------------------------------------------------------------
struct Coef {
    float a, v, b;
};

__device__ __forceinline__ float lambda_of(float w, float r, float beta)
{
    if (!(w > 0.f)) return 1.0f;
    const float x = __fdiv_rn(__fmul_rn(beta, r), __fmul_rn(w, __fsub_rn(1.0f, r)));
    return fminf(fmaxf(x, r), 1.0f);
}

__device__ __forceinline__ Coef coef_of(float w, float r, float beta)
{
    const float lam = lambda_of(w, r, beta);
    Coef c;
    c.a = __fmul_rn(w, __fsub_rn(1.0f, lam));
    const float lw = __fmul_rn(lam, w);
    c.v = __fdiv_rn(__fmul_rn(__fmul_rn(lw, lw), __fsub_rn(1.0f, r)), r);
    c.b = __fmul_rn(__fdiv_rn(lw, r), fmaxf(r, __fsub_rn(1.0f, r)));
    return c;
}

__device__ __forceinline__ float cert_f(float sa, float sv, float bmax, float ld, float D)
{
    const float t = bmax * ld / 3.0f;
    return (sa + t + sqrtf(t * t + 2.0f * sv * ld)) / D;
}

__global__ void __launch_bounds__(1024) beta_kernel(Views views, DecodeArgs a, RowState* __restrict__ rows,
                                                    const float* __restrict__ wl)
{
    __shared__ ff red[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    const int row = blockIdx.x;
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    const SlotView& V = views.v[b];
    RowState& R = rows[row];
    const int nl = R.n_l;
    const float* w = wl + (int64_t)row * a.ws_n;
    const float* rr = V.rl + (int64_t)kv * V.n;
    double lo = 0.0, hi = R.alpha_sum, theta = hi;
    for (int it = 0; it < 200 && nl > 0; ++it) {
        ff A = {0.f, 0.f}, W = {0.f, 0.f}, Rs = {0.f, 0.f};
        for (int j = threadIdx.x; j < nl; j += blockDim.x) {
            const float wj = w[j], rj = rr[j];
            if (!(wj > 0.f)) continue;
            const float al = __fmul_rn(wj, __fsub_rn(1.0f, rj));
            const float ga = __fdiv_rn(al, rj);
            if (theta <= (double)al) A = ff_add_f(A, al);
            else if (theta < (double)ga) {
                W = ff_add_f(W, wj);
                Rs = ff_add_f(Rs, __fdiv_rn(rj, __fsub_rn(1.0f, rj)));
            }
        }
        A = block_sum_ff(A, red);
        W = block_sum_ff(W, red);
        Rs = block_sum_ff(Rs, red);
        const double Ad = ff_to_double(A), Wd = ff_to_double(W), Rd = ff_to_double(Rs);
        const double g = theta * (1.0 + Rd) - Ad - Wd;
        if (g >= 0.0) hi = fmin(hi, theta); else lo = fmax(lo, theta);
        double nt = (Ad + Wd) / (1.0 + Rd);
        if (nt == theta) break;
        if (!(nt > lo && nt < hi)) nt = 0.5 * (lo + hi);
        if (nt == theta || hi - lo <= 1e-16 * hi) { theta = nt; break; }
        theta = nt;
    }
    const double beta = nl > 0 ? theta : 0.0;
    const float bf = (float)beta;
    ff sa = {0.f, 0.f}, sv = {0.f, 0.f};
    float b1 = 0.f, b2 = 0.f;
    int arg = 0x7fffffff;
    for (int j = threadIdx.x; j < nl; j += blockDim.x) {
        const Coef c = coef_of(w[j], rr[j], bf);
        sa = ff_add_f(sa, c.a);
        sv = ff_add_f(sv, c.v);
        if (c.b > b1 || (c.b == b1 && j < arg)) { b2 = b1; b1 = c.b; arg = j; }
        else if (c.b > b2) b2 = c.b;
    }
    sa = block_sum_ff(sa, red);
    sv = block_sum_ff(sv, red);
    // top-2 of b with the argmax (lowest index among equal maxima)
    const float B1 = block_max(b1, redf);
    int cand = (b1 == B1) ? arg : 0x7fffffff;
    __syncthreads();
    {
        int v = cand;
        for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
        if ((threadIdx.x & 31) == 0) redi[threadIdx.x >> 5] = v;
        __syncthreads();
        v = (threadIdx.x & 31) < (blockDim.x >> 5) ? redi[threadIdx.x & 31] : 0x7fffffff;
        for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
        cand = v;
    }
    const int ARG = cand;
    // second largest over everything except ARG
    const float mine2 = (arg == ARG) ? b2 : b1;
    const float B2 = block_max(mine2, redf);
    if (threadIdx.x == 0) {
        const double ld = a.ldelta;
        const double SA = ff_to_double(sa), SV = ff_to_double(sv);
        const double t = (double)B1 * ld / 3.0;
        const double eh = nl > 0 ? (SA + t + sqrt(t * t + 2.0 * SV * ld)) / R.D : 0.0;
        R.beta = beta;
        R.sum_a = SA;
        R.V = SV;
        R.b1 = nl > 0 ? B1 : 0.0;
        R.b2 = nl > 1 ? B2 : 0.0;
        R.b_arg = nl > 0 ? ARG : -1;
        R.eps_hat = eh;
        R.no_fetch = eh < a.eps;
        R.kstar = 0;
        R.fallback = 0;
        R.n_fetch = 0;
    }
}

// --------------------------------------------------------------------------------------------
// D4-D6: gains (eq. (9)), ranking and k* (eq. (10)).  g_i = eps^(L) - eps^(L \ {i}) with lambda
// and D held fixed, written without cancellation:
//   D g_i = a_i + (b - b_-i) l/3 + dA_i / (sqrt(A) + sqrt(A - dA_i)),
//   A = (b l/3)^2 + 2 V l,  dA_i = (b l/3)^2 - (b_-i l/3)^2 + 2 v_i l.
// Keys sort ascending as (g descending, token ascending): key = (~bits(D g)) << 32 | L index.
// The smallest `kSelWidth` keys are found by an MSD radix select (8-bit digits), sorted on chip
// (bitonic), and the certificate of every residual L_g[k:] is evaluated from suffix sums (tail
// of the unsorted rest included).  A row whose k* lies beyond the candidates is flagged for the
// full-row path.
// --------------------------------------------------------------------------------------------
struct GainParams {
    float t;      // b l / 3
    float tm2;    // (b_2 l / 3)
    float sqrtA;
    float A;
    float ld2;    // 2 l
};

__device__ __forceinline__ float gain_num(const Coef& c, int j, int arg, const GainParams& p)
{
    const float tm = (j == arg) ? p.tm2 : p.t;
    const float dA = __fadd_rn(__fsub_rn(__fmul_rn(p.t, p.t), __fmul_rn(tm, tm)), __fmul_rn(p.ld2, c.v));
    const float den = __fadd_rn(p.sqrtA, sqrtf(fmaxf(__fsub_rn(p.A, dA), 0.f)));
    const float root = den > 0.f ? __fdiv_rn(dA, den) : 0.f;
    return fmaxf(__fadd_rn(__fadd_rn(c.a, __fsub_rn(p.t, tm)), root), 0.f);
}

__device__ __forceinline__ GainParams gain_params(const RowState& R, double ld)
{
    GainParams p;
    const double t = R.b1 * ld / 3.0, t2 = R.b2 * ld / 3.0;
    const double A = t * t + 2.0 * R.V * ld;
    p.t = (float)t;
    p.tm2 = (float)t2;
    p.A = (float)A;
    p.sqrtA = (float)sqrt(A);
    p.ld2 = (float)(2.0 * ld);
    return p;
}

__device__ __forceinline__ unsigned long long gain_key(float gnum, int j)
{
    return ((unsigned long long)(~__float_as_uint(gnum)) << 32) | (unsigned)j;
}

// Block-wide inclusive scan (float-float sums + running max) in reverse thread order.
struct ScanVal {
    ff a, v;
    float b;
};

__device__ __forceinline__ ScanVal scan_combine(const ScanVal& x, const ScanVal& y)
{
    return {ff_add(x.a, y.a), ff_add(x.v, y.v), fmaxf(x.b, y.b)};
}

// Returns the sum over threads with index > threadIdx.x (exclusive suffix).
__device__ ScanVal block_suffix_exclusive(ScanVal mine, ScanVal* sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    // inclusive suffix within warp: combine with lanes above
    ScanVal x = mine;
    for (int o = 1; o < 32; o <<= 1) {
        ScanVal y;
        y.a.hi = __shfl_down_sync(0xffffffffu, x.a.hi, o);
        y.a.lo = __shfl_down_sync(0xffffffffu, x.a.lo, o);
        y.v.hi = __shfl_down_sync(0xffffffffu, x.v.hi, o);
        y.v.lo = __shfl_down_sync(0xffffffffu, x.v.lo, o);
        y.b = __shfl_down_sync(0xffffffffu, x.b, o);
        if (lane + o < 32) x = scan_combine(x, y);
    }
    __syncthreads();
    if (lane == 0) sh[warp] = x;  // whole-warp total
    __syncthreads();
    ScanVal after = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
    for (int w2 = warp + 1; w2 < nw; ++w2) after = scan_combine(after, sh[w2]);
    // exclusive within warp: inclusive minus own = inclusive of lane + 1
    ScanVal nxt;
    nxt.a.hi = __shfl_down_sync(0xffffffffu, x.a.hi, 1);
    nxt.a.lo = __shfl_down_sync(0xffffffffu, x.a.lo, 1);
    nxt.v.hi = __shfl_down_sync(0xffffffffu, x.v.hi, 1);
    nxt.v.lo = __shfl_down_sync(0xffffffffu, x.v.lo, 1);
    nxt.b = __shfl_down_sync(0xffffffffu, x.b, 1);
    if (lane == 31) nxt = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
    return scan_combine(nxt, after);
}

__device__ __forceinline__ void bitonic_sort_smem(unsigned long long* k, int P)
{
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = ((lo & size) == 0);
                const unsigned long long x = k[lo], y = k[hi];
                if ((x > y) == up) { k[lo] = y; k[hi] = x; }
            }
        }
    }
    __syncthreads();
}

// Write E_h = the first k* entries of the sorted keys.
__device__ void emit_exact_set(const unsigned long long* sorted, int kstar, int row, const SlotView& V, int kv,
                               DecodeArgs a, int32_t* __restrict__ mark, int32_t* __restrict__ elist,
                               RowState& R, int* redi)
{
    int nf = 0;
    for (int p = threadIdx.x; p < kstar; p += blockDim.x) {
        const int j = (int)(sorted[p] & 0xffffffffu);
        const int tok = V.ltok[(int64_t)kv * V.n + j];
        mark[(int64_t)row * a.ws_n + j] = a.gen;
        elist[(int64_t)row * a.ws_n + p] = tok;
        nf += V.flags[(int64_t)kv * V.n + tok] == 0;
    }
    nf = block_sum(nf, redi);
    if (threadIdx.x == 0) {
        R.kstar = kstar;
        R.n_fetch = nf;
    }
}

__global__ void __launch_bounds__(1024) select_kernel(Views views, DecodeArgs a, RowState* __restrict__ rows,
                                                      const float* __restrict__ wl,
                                                      unsigned long long* __restrict__ keys,
                                                      int32_t* __restrict__ mark, int32_t* __restrict__ elist)
{
    extern __shared__ unsigned long long cand[];  // [kSelWidth]
    __shared__ int hist[256];
    __shared__ ScanVal shs[32];
    __shared__ ff redff[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ int ccount;
    __shared__ int sel_digit, sel_need, sel_all;
    __shared__ int best_k;
    const int row = blockIdx.x;
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    const SlotView& V = views.v[b];
    RowState& R = rows[row];
    if (R.no_fetch) return;
    const int nl = R.n_l;
    const float* w = wl + (int64_t)row * a.ws_n;
    const float* rr = V.rl + (int64_t)kv * V.n;
    unsigned long long* key = keys + (int64_t)row * a.ws_npow2;
    const float bf = (float)R.beta;
    const GainParams gp = gain_params(R, a.ldelta);
    const int arg = R.b_arg;
    for (int j = threadIdx.x; j < nl; j += blockDim.x) {
        const Coef c = coef_of(w[j], rr[j], bf);
        key[j] = gain_key(gain_num(c, j, arg, gp), j);
    }
    // --- radix select of the kSelWidth smallest keys
    unsigned long long T = ~0ull;
    if (nl > kSelWidth) {
        unsigned long long prefix = 0, pmask = 0;
        int need = kSelWidth;
        bool done = false;
        for (int shift = 56; shift >= 0 && !done; shift -= 8) {
            __syncthreads();
            for (int d = threadIdx.x; d < 256; d += blockDim.x) hist[d] = 0;
            __syncthreads();
            for (int j = threadIdx.x; j < nl; j += blockDim.x) {
                const unsigned long long k = key[j];
                if ((k & pmask) == prefix) {
                    const unsigned dig = (unsigned)((k >> shift) & 255);
                    const unsigned peers = __match_any_sync(__activemask(), dig);
                    if ((__ffs(peers) - 1) == (threadIdx.x & 31)) atomicAdd(&hist[dig], __popc(peers));
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                int cum = 0, d = 0;
                for (d = 0; d < 255; ++d) {
                    if (cum + hist[d] >= need) break;
                    cum += hist[d];
                }
                sel_digit = d;
                sel_need = need - cum;
                sel_all = hist[d] == need - cum;
            }
            __syncthreads();
            prefix |= (unsigned long long)sel_digit << shift;
            pmask |= 255ull << shift;
            need = sel_need;
            done = sel_all;
        }
        T = done ? (prefix | ~pmask) : prefix;
    }
    // --- gather candidates (key <= T) and the tail sums of the rest
    if (threadIdx.x == 0) ccount = 0;
    __syncthreads();
    ff ta = {0.f, 0.f}, tv = {0.f, 0.f};
    float tb = 0.f;
    for (int j = threadIdx.x; j < nl; j += blockDim.x) {
        const unsigned long long k = key[j];
        if (k <= T) {
            const int pos = atomicAdd(&ccount, 1);
            cand[pos] = k;
        } else {
            const Coef c = coef_of(w[j], rr[j], bf);
            ta = ff_add_f(ta, c.a);
            tv = ff_add_f(tv, c.v);
            tb = fmaxf(tb, c.b);
        }
    }
    ta = block_sum_ff(ta, redff);
    tv = block_sum_ff(tv, redff);
    tb = block_max(tb, redf);
    __syncthreads();
    const int cnt = ccount;
    int P = 1;
    while (P < cnt) P <<= 1;
    for (int p = cnt + threadIdx.x; p < P; p += blockDim.x) cand[p] = ~0ull;
    bitonic_sort_smem(cand, P);
    // --- suffix sums over the sorted candidates; thread t owns a contiguous chunk
    const int per = (cnt + blockDim.x - 1) / blockDim.x;
    const int p0 = min(cnt, (int)threadIdx.x * per), p1 = min(cnt, p0 + per);
    ScanVal mine = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
    for (int p = p0; p < p1; ++p) {
        const int j = (int)(cand[p] & 0xffffffffu);
        const Coef c = coef_of(w[j], rr[j], bf);
        mine = scan_combine(mine, ScanVal{{c.a, 0.f}, {c.v, 0.f}, c.b});
    }
    ScanVal after = block_suffix_exclusive(mine, shs);
    after = scan_combine(after, ScanVal{ta, tv, tb});
    if (threadIdx.x == 0) best_k = 0x7fffffff;
    __syncthreads();
    const float ld = (float)a.ldelta, D = (float)R.D;
    int local_best = 0x7fffffff;
    ScanVal run = after;
    for (int p = p1 - 1; p >= p0; --p) {
        const int j = (int)(cand[p] & 0xffffffffu);
        const Coef c = coef_of(w[j], rr[j], bf);
        run = scan_combine(run, ScanVal{{c.a, 0.f}, {c.v, 0.f}, c.b});
        // run = residual L_g[p:] (this element and everything after it)
        if (p >= 1 && cert_f(run.a.hi + run.a.lo, run.v.hi + run.v.lo, run.b, ld, D) < a.eps_f) local_best = p;
    }
    if (local_best != 0x7fffffff) atomicMin(&best_k, local_best);
    __syncthreads();
    int kstar = best_k;
    if (kstar == 0x7fffffff) {
        // removing every candidate: only the tail remains
        if (cnt == nl || cert_f(ta.hi + ta.lo, tv.hi + tv.lo, tb, ld, D) < a.eps_f) kstar = cnt;
    }
    if (kstar == 0x7fffffff) {
        if (threadIdx.x == 0) { R.fallback = 1; R.kstar = -1; }
        return;
    }
    emit_exact_set(cand, kstar, row, V, kv, a, mark, elist, R, redi);
}

// Full-row path: bitonic sort of every key in global memory, then the residual certificates from
// the end of the order backwards until the first one that is not below eps.
__global__ void __launch_bounds__(1024) fallback_kernel(Views views, DecodeArgs a, RowState* __restrict__ rows,
                                                        const float* __restrict__ wl,
                                                        unsigned long long* __restrict__ keys,
                                                        int32_t* __restrict__ mark, int32_t* __restrict__ elist)
{
    __shared__ ScanVal shs[32];
    __shared__ int redi[32];
    __shared__ int found;
    const int row = blockIdx.x;
    RowState& R = rows[row];
    if (!R.fallback) return;
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    const SlotView& V = views.v[b];
    const int nl = R.n_l;
    const float* w = wl + (int64_t)row * a.ws_n;
    const float* rr = V.rl + (int64_t)kv * V.n;
    unsigned long long* key = keys + (int64_t)row * a.ws_npow2;
    const float bf = (float)R.beta;
    int P = 1;
    while (P < nl) P <<= 1;
    for (int p = nl + threadIdx.x; p < P; p += blockDim.x) key[p] = ~0ull;
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool up = ((lo & size) == 0);
                const unsigned long long x = key[lo], y = key[hi];
                if ((x > y) == up) { key[lo] = y; key[hi] = x; }
            }
            __syncthreads();
        }
    }
    const float ld = (float)a.ldelta, D = (float)R.D;
    __shared__ ScanVal chunk_total;
    ScanVal carry = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
    if (threadIdx.x == 0) found = -1;
    __syncthreads();
    int kstar = -1;
    for (int c1 = nl; c1 > 0; c1 -= blockDim.x) {
        const int c0 = max(0, c1 - (int)blockDim.x);
        const int p = c0 + threadIdx.x;
        ScanVal mine = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
        if (p < c1) {
            const int j = (int)(key[p] & 0xffffffffu);
            const Coef c = coef_of(w[j], rr[j], bf);
            mine = ScanVal{{c.a, 0.f}, {c.v, 0.f}, c.b};
        }
        const ScanVal after = block_suffix_exclusive(mine, shs);
        const ScanVal own = scan_combine(mine, after);
        const ScanVal incl = scan_combine(own, carry);  // residual L_g[p:]
        if (p < c1 && p >= 1 && !(cert_f(incl.a.hi + incl.a.lo, incl.v.hi + incl.v.lo, incl.b, ld, D) < a.eps_f))
            atomicMax(&found, p);
        if (threadIdx.x == 0) chunk_total = own;
        __syncthreads();
        if (found >= 0) { kstar = found + 1; break; }
        carry = scan_combine(carry, chunk_total);
        __syncthreads();
    }
    if (kstar < 1) kstar = 1;
    if (threadIdx.x == 0) R.fallback = 1;
    emit_exact_set(key, kstar, row, V, kv, a, mark, elist, R, redi);
}

// --------------------------------------------------------------------------------------------
// D7: union of L_g[:k*] \ S over the query heads of a KV head (ascending tokens), and the copy of
// those rows from the pinned host cache into the staging area (zero-copy loads, one warp per
// row, 16 bytes per lane).
// --------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) union_kernel(Views views, DecodeArgs a, const RowState* __restrict__ rows,
                                                     const int32_t* __restrict__ elist, uint32_t* __restrict__ ubits,
                                                     int32_t* __restrict__ ulist, int32_t* __restrict__ ucount)
{
    __shared__ int scratch[32];
    const int b = blockIdx.x / a.Hkv, kv = blockIdx.x % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int nwords = (n + 31) / 32;
    uint32_t* bits = ubits + (int64_t)(b * a.Hkv + kv) * (a.ws_n / 32 + 1);
    for (int g = 0; g < a.G; ++g) {
        const int row = row_of(b, kv * a.G + g, a.Hq);
        const int ks = rows[row].kstar;
        for (int p = threadIdx.x; p < ks; p += blockDim.x) {
            const int tok = elist[(int64_t)row * a.ws_n + p];
            if (V.flags[(int64_t)kv * n + tok] == 0) atomicOr(&bits[tok >> 5], 1u << (tok & 31));
        }
    }
    __syncthreads();
    int base = 0;
    int32_t* out = ulist + (int64_t)(b * a.Hkv + kv) * a.ws_n;
    for (int w0 = 0; w0 < nwords; w0 += blockDim.x) {
        const int wi = w0 + threadIdx.x;
        uint32_t word = wi < nwords ? bits[wi] : 0u;
        int total;
        const int ex = block_exclusive_scan(__popc(word), scratch, &total);
        int pos = base + ex;
        if (wi < nwords && word) {
            bits[wi] = 0u;
            while (word) {
                const int bit = __ffs(word) - 1;
                out[pos++] = wi * 32 + bit;
                word &= word - 1;
            }
        }
        base += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) ucount[b * a.Hkv + kv] = base;
}

__global__ void gather_kernel(Views views, DecodeArgs a, const int32_t* __restrict__ ulist,
                              const int32_t* __restrict__ ucount, unsigned char* __restrict__ staging, int row_bytes)
{
    const int b = blockIdx.x / a.Hkv, kv = blockIdx.x % a.Hkv;
    const SlotView& V = views.v[b];
    const int cnt = ucount[b * a.Hkv + kv];
    const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
    const int32_t* lst = ulist + (int64_t)(b * a.Hkv + kv) * a.ws_n;
    const unsigned char* host = reinterpret_cast<const unsigned char*>(V.kv_host);
    unsigned char* dst = staging + (int64_t)(b * a.Hkv + kv) * a.ws_n * row_bytes;
    for (int u = blockIdx.y * warps + (threadIdx.x >> 5); u < cnt; u += gridDim.y * warps) {
        const int tok = lst[u];
        const uint4* src = reinterpret_cast<const uint4*>(host + ((int64_t)kv * V.n + tok) * row_bytes);
        uint4* to = reinterpret_cast<uint4*>(dst + (int64_t)u * row_bytes);
        for (int v = lane; v < row_bytes / 16; v += 32) to[v] = src[v];
    }
}

// --------------------------------------------------------------------------------------------
// D8: weighted attention (comment closing Algorithm 2; estimator of Theorem 2).  Rows: the
// resident H u S rows and the staged rows of the KV head; per query head the weight factor is 1 on
// H and on L_g[:k*], lambda_i / r_i on S \ L_g[:k*], and 0 on staged rows fetched for another query
// head.  Split over `nsplit` blocks per KV head; one warp per K/V row, 4 channels per lane, all G
// query heads at once (each K/V byte is read once for the group).
// --------------------------------------------------------------------------------------------
template <typename T> struct Vec4;
template <> struct Vec4<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load(const __nv_bfloat16* p)
    {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
        const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
        const float2 fx = __bfloat1622float2(x), fy = __bfloat1622float2(y);
        return make_float4(fx.x, fx.y, fy.x, fy.y);
    }
};
template <> struct Vec4<float> {
    static __device__ __forceinline__ float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
};

template <typename T, int G>
__global__ void __launch_bounds__(128) attn_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                   const RowState* __restrict__ rows, const float* __restrict__ wl,
                                                   const int32_t* __restrict__ mark,
                                                   const int32_t* __restrict__ ulist, const int32_t* __restrict__ ucount,
                                                   const T* __restrict__ staging, float* __restrict__ part)
{
    __shared__ float sm_m[4][G], sm_l[4][G];
    __shared__ float sm_acc[4][G][kHeadDim];
    const int b = blockIdx.x / a.Hkv, kv = blockIdx.x % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m_res = V.counts[kv * 4 + 3];
    const int nu = ucount[b * a.Hkv + kv];
    const int total = m_res + nu;
    const int per = (total + a.nsplit - 1) / a.nsplit;
    const int r0 = blockIdx.y * per, r1 = min(total, r0 + per);
    float qv[G][4];
    float beta[G];
    int rowg[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        rowg[g] = row_of(b, kv * G + g, a.Hq);
        const float4 t = *reinterpret_cast<const float4*>(q + (int64_t)rowg[g] * kHeadDim + lane * 4);
        qv[g][0] = t.x; qv[g][1] = t.y; qv[g][2] = t.z; qv[g][3] = t.w;
        beta[g] = (float)rows[rowg[g]].beta;
    }
    float mrun[G], lrun[G], acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        mrun[g] = -INFINITY;
        lrun[g] = 0.f;
        acc[g][0] = acc[g][1] = acc[g][2] = acc[g][3] = 0.f;
    }
    const T* res = reinterpret_cast<const T*>(V.kvres) + V.res_off[kv] * 2 * kHeadDim;
    const T* stg = staging + (int64_t)(b * a.Hkv + kv) * a.ws_n * 2 * kHeadDim;
    for (int rix = r0 + warp; rix < r1; rix += 4) {
        const T* rowp;
        int tok;
        bool staged = rix >= m_res;
        if (!staged) {
            rowp = res + (int64_t)rix * 2 * kHeadDim;
            tok = V.rtok[(int64_t)kv * n + rix];
        } else {
            const int u = rix - m_res;
            rowp = stg + (int64_t)u * 2 * kHeadDim;
            tok = ulist[(int64_t)(b * a.Hkv + kv) * a.ws_n + u];
        }
        const int f = V.flags[(int64_t)kv * n + tok];
        const int li = V.lpos[(int64_t)kv * n + tok];
        const float4 k4 = Vec4<T>::load(rowp + lane * 4);
        const float4 v4 = Vec4<T>::load(rowp + kHeadDim + lane * 4);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float s = qv[g][0] * k4.x + qv[g][1] * k4.y + qv[g][2] * k4.z + qv[g][3] * k4.w;
            s = warp_sum(s);
            float om;
            if (f == 2) om = 1.f;
            else {
                const bool exact = mark[(int64_t)rowg[g] * a.ws_n + li] == a.gen;
                if (exact) om = 1.f;
                else if (f == 1 && !staged) {
                    const float r = V.rl[(int64_t)kv * n + li];
                    om = __fdiv_rn(lambda_of(wl[(int64_t)rowg[g] * a.ws_n + li], r, beta[g]), r);
                } else om = 0.f;
            }
            if (om > 0.f) {
                const float x = s * a.inv_sqrt_d_f;
                const float mn = fmaxf(mrun[g], x);
                const float corr = expf(mrun[g] - mn);
                const float p = om * expf(x - mn);
                lrun[g] = lrun[g] * corr + p;
                acc[g][0] = acc[g][0] * corr + p * v4.x;
                acc[g][1] = acc[g][1] * corr + p * v4.y;
                acc[g][2] = acc[g][2] * corr + p * v4.z;
                acc[g][3] = acc[g][3] * corr + p * v4.w;
                mrun[g] = mn;
            }
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) { sm_m[warp][g] = mrun[g]; sm_l[warp][g] = lrun[g]; }
        sm_acc[warp][g][lane * 4 + 0] = acc[g][0];
        sm_acc[warp][g][lane * 4 + 1] = acc[g][1];
        sm_acc[warp][g][lane * 4 + 2] = acc[g][2];
        sm_acc[warp][g][lane * 4 + 3] = acc[g][3];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G * kHeadDim; e += blockDim.x) {
        const int g = e / kHeadDim, c = e % kHeadDim;
        float M = -INFINITY;
        for (int w2 = 0; w2 < 4; ++w2) M = fmaxf(M, sm_m[w2][g]);
        float L = 0.f, A = 0.f;
        if (M > -INFINITY)
            for (int w2 = 0; w2 < 4; ++w2) {
                const float s = sm_m[w2][g] > -INFINITY ? expf(sm_m[w2][g] - M) : 0.f;
                L += sm_l[w2][g] * s;
                A += sm_acc[w2][g][c] * s;
            }
        float* pp = part + ((int64_t)rowg[g] * a.nsplit + blockIdx.y) * (kHeadDim + 2);
        pp[c] = A;
        if (c == 0) { pp[kHeadDim] = M; pp[kHeadDim + 1] = L; }
    }
}

__global__ void merge_kernel(DecodeArgs a, const float* __restrict__ part, float* __restrict__ out)
{
    const int row = blockIdx.x, c = threadIdx.x;
    const float* pp = part + (int64_t)row * a.nsplit * (kHeadDim + 2);
    float M = -INFINITY;
    for (int s = 0; s < a.nsplit; ++s) M = fmaxf(M, pp[s * (kHeadDim + 2) + kHeadDim]);
    float L = 0.f, A = 0.f;
    for (int s = 0; s < a.nsplit; ++s) {
        const float m = pp[s * (kHeadDim + 2) + kHeadDim];
        if (m == -INFINITY) continue;
        const float sc = expf(m - M);
        L += pp[s * (kHeadDim + 2) + kHeadDim + 1] * sc;
        A += pp[s * (kHeadDim + 2) + c] * sc;
    }
    out[(int64_t)row * kHeadDim + c] = A / L;
}

template <typename T, int G>
verkv_status launch_decode(Ctx& ctx, const Views& views, const DecodeArgs& a, int B, int max_n, int max_nl,
                           int max_nh, const float* q, float* out, cudaStream_t st)
{
    const verkv_config& cfg = ctx.cfg;
    const int rowsN = B * a.Hq;
    VK_TIMING_BEGIN();
    init_rows_kernel<<<(rowsN + 127) / 128, 128, 0, st>>>(ctx.rows, views, a, B);
    VK_LAUNCHED("init_rows");
    const dim3 gs((max_n + kTile - 1) / kTile, B * a.Hkv);
    if (cfg.sketch == VERKV_SKETCH_INT8)
        score_int8_kernel<G><<<gs, kTile, 0, st>>>(views, q, a, ctx.rows, ctx.tl);
    else if (cfg.sketch == VERKV_SKETCH_2BIT)
        score_2bit_kernel<G><<<gs, kTile, 0, st>>>(views, q, a, ctx.rows, ctx.tl);
    else
        score_exact_kernel<T, G><<<gs, kTile, 0, st>>>(views, q, a, ctx.rows, ctx.tl);
    VK_LAUNCHED("score_sketch");
    if (max_nh > 0) {
        score_h_kernel<T, G><<<dim3((max_nh + kTile - 1) / kTile, B * a.Hkv), kTile, 0, st>>>(views, q, a, ctx.rows,
                                                                                            ctx.th);
        VK_LAUNCHED("score_h");
    }
    const int wmax = std::max(max_nl, max_nh);
    weights_kernel<<<dim3(std::max(1, (wmax + 255) / 256), rowsN), 256, 0, st>>>(views, a, ctx.rows, ctx.tl, ctx.th,
                                                                                ctx.wl);
    VK_LAUNCHED("weights");
    beta_kernel<<<rowsN, 1024, 0, st>>>(views, a, ctx.rows, ctx.wl);
    VK_LAUNCHED("beta");
    const size_t sel_smem = sizeof(unsigned long long) * kSelWidth;
    select_kernel<<<rowsN, 1024, sel_smem, st>>>(views, a, ctx.rows, ctx.wl, ctx.keys, ctx.mark, ctx.elist);
    VK_LAUNCHED("select");
    fallback_kernel<<<rowsN, 1024, 0, st>>>(views, a, ctx.rows, ctx.wl, ctx.keys, ctx.mark, ctx.elist);
    VK_LAUNCHED("fallback");
    union_kernel<<<B * a.Hkv, 1024, 0, st>>>(views, a, ctx.rows, ctx.elist, ctx.ubits, ctx.ulist, ctx.ucount);
    VK_LAUNCHED("union");
    const int row_bytes = (int)(2 * kHeadDim * sizeof(T));
    gather_kernel<<<dim3(B * a.Hkv, 16), 256, 0, st>>>(views, a, ctx.ulist, ctx.ucount,
                                                       (unsigned char*)ctx.staging, row_bytes);
    VK_LAUNCHED("gather");
    attn_kernel<T, G><<<dim3(B * a.Hkv, a.nsplit), 128, 0, st>>>(views, q, a, ctx.rows, ctx.wl, ctx.mark, ctx.ulist,
                                                                 ctx.ucount, (const T*)ctx.staging, ctx.part);
    VK_LAUNCHED("attn");
    merge_kernel<<<rowsN, kHeadDim, 0, st>>>(a, ctx.part, out);
    VK_LAUNCHED("merge");
    return VERKV_OK;
}

template <typename T>
verkv_status dispatch_g(Ctx& ctx, const Views& views, const DecodeArgs& a, int B, int max_n, int max_nl, int max_nh,
                        const float* q, float* out, cudaStream_t st)
{
    switch (ctx.G) {
        case 1: return launch_decode<T, 1>(ctx, views, a, B, max_n, max_nl, max_nh, q, out, st);
        case 2: return launch_decode<T, 2>(ctx, views, a, B, max_n, max_nl, max_nh, q, out, st);
        case 4: return launch_decode<T, 4>(ctx, views, a, B, max_n, max_nl, max_nh, q, out, st);
        case 8: return launch_decode<T, 8>(ctx, views, a, B, max_n, max_nl, max_nh, q, out, st);
        default: ctx.err = "GQA group must be 1, 2, 4 or 8"; return VERKV_EUNSUPPORTED;
    }
}

bool g_attr_done = false;

}  // namespace

int decode_max_batch() { return kMaxBatch; }
int decode_sel_width() { return kSelWidth; }

verkv_status decode_rows(Ctx& ctx, int layer, const int32_t* seq_ids, int B, const float* q, double eps,
                         double delta, float* out, cudaStream_t st)
{
    const verkv_config& cfg = ctx.cfg;
    if (B > kMaxBatch) {
        ctx.err = "batch larger than the built maximum";
        return VERKV_EINVAL;
    }
    if (!g_attr_done) {
        VK_CUDA(cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(sizeof(unsigned long long) * kSelWidth)));
        g_attr_done = true;
    }
    Views views;
    memset(&views, 0, sizeof(views));
    int max_n = 0, max_nl = 0, max_nh = 0;
    ctx.last_seq.assign(seq_ids, seq_ids + B);
    ctx.last_n.clear();
    for (int b = 0; b < B; ++b) {
        Slot& s = ctx.slot(layer, seq_ids[b]);
        SlotView& v = views.v[b];
        v.n = s.n;
        v.r = s.r;
        v.flags = s.flags;
        v.lpos = s.lpos;
        v.ltok = s.ltok;
        v.rl = s.rl;
        v.rtok = s.rtok;
        v.hslot = s.hslot;
        v.counts = s.counts;
        v.kvres = s.kvres;
        v.res_off = s.res_off;
        v.kv_host = s.kv_host;
        v.codes8 = s.codes8;
        v.scale8 = s.scale8;
        v.codes2 = s.codes2;
        v.zero2 = s.zero2;
        v.scale2 = s.scale2;
        v.pairs = s.pairs;
        v.kexact = s.kexact;
        max_n = std::max(max_n, s.n);
        for (const verkv_head_stats& hs : s.stats) {
            max_nl = std::max(max_nl, hs.n_l);
            max_nh = std::max(max_nh, hs.n_h);
        }
        ctx.last_n.push_back(s.n);
    }
    DecodeArgs a;
    a.Hkv = cfg.n_kv_heads;
    a.Hq = cfg.n_q_heads;
    a.G = ctx.G;
    a.ws_n = ctx.ws_n;
    a.ws_npow2 = ctx.ws_npow2;
    a.gen = ++ctx.gen;
    a.nsplit = ctx.nsplit;
    a.eps = eps;
    a.eps_f = (float)eps;
    a.ldelta = std::log(2.0 / delta);
    const double isd = 1.0 / std::sqrt((double)kHeadDim);
    a.inv_sqrt_d_f = (float)isd;
    a.inv_sqrt_d.hi = (float)isd;
    a.inv_sqrt_d.lo = (float)(isd - (double)(float)isd);
    ctx.last_launches = 0;
    ctx.last_B = B;
    ctx.last_layer = layer;
    if (cfg.kv_dtype == VERKV_DTYPE_BF16)
        return dispatch_g<__nv_bfloat16>(ctx, views, a, B, max_n, max_nl, max_nh, q, out, st);
    return dispatch_g<float>(ctx, views, a, B, max_n, max_nl, max_nh, q, out, st);
}

}  // namespace verkv

// ================================================================================================
// Allocation-free variant of the per-row decision (the beta solve, eq. (7), the gains, the full-row
// ranking and k* of the full-row path above) for callers that cannot allocate device memory: code
// running where cudaMalloc is unavailable or forbidden (inside a stream capture whose graph must not
// own allocations, under an external memory pool or budget, in a real-time loop).  Its only scratch
// is the file-scope array below, which every GPU that loads the library holds until the process
// exits; all calls share it.
// ================================================================================================
#include <mutex>

namespace verkv {
namespace {

constexpr int kStaticMaxL = 65536;  // largest |L| the allocation-free entry point accepts
__device__ __align__(256) unsigned long long g_static_keys[kStaticMaxL];

__global__ void __launch_bounds__(1024) certify_static_kernel(const float* __restrict__ w, const float* __restrict__ rr,
                                                              int nl, double D, float eps_f, double eps, double ld,
                                                              unsigned long long* __restrict__ key,
                                                              double* __restrict__ out_scalars,
                                                              int32_t* __restrict__ out_kstar,
                                                              int32_t* __restrict__ out_exact)
{
    __shared__ ff red[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ ScanVal shs[32];
    __shared__ ScanVal chunk_total;
    __shared__ int found;
    // top of the beta bracket: sum_L w (1 - r)
    ff al = {0.f, 0.f};
    for (int j = threadIdx.x; j < nl; j += blockDim.x) al = ff_add(al, two_prod(w[j], __fsub_rn(1.0f, rr[j])));
    al = block_sum_ff(al, red);
    double lo = 0.0, hi = ff_to_double(al), theta = hi;
    // safeguarded Newton on G(beta) = beta (1 + R) - A - W (Definition 2's fixed point)
    for (int it = 0; it < 200 && nl > 0; ++it) {
        ff A = {0.f, 0.f}, Wf = {0.f, 0.f}, Rs = {0.f, 0.f};
        for (int j = threadIdx.x; j < nl; j += blockDim.x) {
            const float wj = w[j], rj = rr[j];
            if (!(wj > 0.f)) continue;
            const float a1 = __fmul_rn(wj, __fsub_rn(1.0f, rj));
            const float ga = __fdiv_rn(a1, rj);
            if (theta <= (double)a1) A = ff_add_f(A, a1);
            else if (theta < (double)ga) {
                Wf = ff_add_f(Wf, wj);
                Rs = ff_add_f(Rs, __fdiv_rn(rj, __fsub_rn(1.0f, rj)));
            }
        }
        A = block_sum_ff(A, red);
        Wf = block_sum_ff(Wf, red);
        Rs = block_sum_ff(Rs, red);
        const double Ad = ff_to_double(A), Wd = ff_to_double(Wf), Rd = ff_to_double(Rs);
        const double g = theta * (1.0 + Rd) - Ad - Wd;
        if (g >= 0.0) hi = fmin(hi, theta); else lo = fmax(lo, theta);
        double nt = (Ad + Wd) / (1.0 + Rd);
        if (nt == theta) break;
        if (!(nt > lo && nt < hi)) nt = 0.5 * (lo + hi);
        if (nt == theta || hi - lo <= 1e-16 * hi) { theta = nt; break; }
        theta = nt;
    }
    const double beta = nl > 0 ? theta : 0.0;
    const float bf = (float)beta;
    // eq. (7) sums and the two largest b_i
    ff sa = {0.f, 0.f}, sv = {0.f, 0.f};
    float b1 = 0.f, b2 = 0.f;
    int arg = 0x7fffffff;
    for (int j = threadIdx.x; j < nl; j += blockDim.x) {
        const Coef c = coef_of(w[j], rr[j], bf);
        sa = ff_add_f(sa, c.a);
        sv = ff_add_f(sv, c.v);
        if (c.b > b1 || (c.b == b1 && j < arg)) { b2 = b1; b1 = c.b; arg = j; }
        else if (c.b > b2) b2 = c.b;
    }
    sa = block_sum_ff(sa, red);
    sv = block_sum_ff(sv, red);
    const float B1 = block_max(b1, redf);
    int cand = (b1 == B1) ? arg : 0x7fffffff;
    __syncthreads();
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    if ((threadIdx.x & 31) == 0) redi[threadIdx.x >> 5] = cand;
    __syncthreads();
    cand = (threadIdx.x & 31) < (blockDim.x >> 5) ? redi[threadIdx.x & 31] : 0x7fffffff;
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    const int ARG = cand;
    const float B2 = block_max((arg == ARG) ? b2 : b1, redf);
    const double SA = ff_to_double(sa), SV = ff_to_double(sv);
    const double t = (double)B1 * ld / 3.0;
    const double eh = nl > 0 ? (SA + t + sqrt(t * t + 2.0 * SV * ld)) / D : 0.0;
    const bool no_fetch = eh < eps;
    if (threadIdx.x == 0) {
        out_scalars[0] = beta;
        out_scalars[1] = eh;
        out_scalars[2] = SA;
        out_scalars[3] = SV;
    }
    if (no_fetch) {
        if (threadIdx.x == 0) *out_kstar = 0;
        return;
    }
    // gains (eq. (9)) as sort keys: (g descending, index ascending)
    GainParams gp;
    {
        const double t2 = (nl > 1 ? (double)B2 : 0.0) * ld / 3.0;
        const double Aq = t * t + 2.0 * SV * ld;
        gp.t = (float)t;
        gp.tm2 = (float)t2;
        gp.A = (float)Aq;
        gp.sqrtA = (float)sqrt(Aq);
        gp.ld2 = (float)(2.0 * ld);
    }
    int P = 1;
    while (P < nl) P <<= 1;
    for (int j = threadIdx.x; j < P; j += blockDim.x) {
        if (j < nl) {
            const Coef c = coef_of(w[j], rr[j], bf);
            key[j] = gain_key(gain_num(c, j, ARG, gp), j);
        } else {
            key[j] = ~0ull;  // padding: every call rewrites [0, P)
        }
    }
    __syncthreads();
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
                const int a0 = 2 * i - (i & (stride - 1));
                const int a1 = a0 + stride;
                const bool up = ((a0 & size) == 0);
                const unsigned long long x = key[a0], y = key[a1];
                if ((x > y) == up) { key[a0] = y; key[a1] = x; }
            }
            __syncthreads();
        }
    }
    // eq. (10): residual certificates from the end of the order backwards
    const float ldf = (float)ld, Df = (float)D;
    ScanVal carry = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
    if (threadIdx.x == 0) found = -1;
    __syncthreads();
    int kstar = -1;
    for (int c1 = nl; c1 > 0; c1 -= blockDim.x) {
        const int c0 = max(0, c1 - (int)blockDim.x);
        const int p = c0 + threadIdx.x;
        ScanVal mine = {{0.f, 0.f}, {0.f, 0.f}, 0.f};
        if (p < c1) {
            const int j = (int)(key[p] & 0xffffffffu);
            const Coef c = coef_of(w[j], rr[j], bf);
            mine = ScanVal{{c.a, 0.f}, {c.v, 0.f}, c.b};
        }
        const ScanVal after = block_suffix_exclusive(mine, shs);
        const ScanVal own = scan_combine(mine, after);
        const ScanVal incl = scan_combine(own, carry);
        if (p < c1 && p >= 1 && !(cert_f(incl.a.hi + incl.a.lo, incl.v.hi + incl.v.lo, incl.b, ldf, Df) < eps_f))
            atomicMax(&found, p);
        if (threadIdx.x == 0) chunk_total = own;
        __syncthreads();
        if (found >= 0) { kstar = found + 1; break; }
        carry = scan_combine(carry, chunk_total);
        __syncthreads();
    }
    if (kstar < 1) kstar = 1;
    for (int p = threadIdx.x; p < kstar; p += blockDim.x) out_exact[p] = (int32_t)(key[p] & 0xffffffffu);
    if (threadIdx.x == 0) *out_kstar = kstar;
}

std::mutex g_static_mu;
void* g_static_ptr[256] = {};

}  // namespace
}  // namespace verkv

extern "C" verkv_status verkv_certify_row_static(const float* w_hat, const float* r, int32_t n_l, double D, double eps,
                                                 double delta, double* scalars, int32_t* kstar, int32_t* exact,
                                                 verkv_stream stream)
{
    using namespace verkv;
    if (n_l < 0 || n_l > kStaticMaxL) return VERKV_EINVAL;  // beyond the static scratch
    if (!(eps >= 0.0) || !std::isfinite(eps) || !(delta > 0.0 && delta < 1.0) || !(D > 0.0)) return VERKV_EINVAL;
    if (!scalars || !kstar || (n_l > 0 && (!w_hat || !r || !exact))) return VERKV_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return VERKV_ECUDA;
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_static_mu);
        if (!g_static_ptr[dev]) {
            // the array's host-side name is only a stand-in: its device address comes from the runtime
            if (cudaGetSymbolAddress(&g_static_ptr[dev], g_static_keys) != cudaSuccess) {
                g_static_ptr[dev] = nullptr;
                return VERKV_ECUDA;
            }
        }
        ptr = g_static_ptr[dev];
    }
    certify_static_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(
        w_hat, r, n_l, D, (float)eps, eps, std::log(2.0 / delta), reinterpret_cast<unsigned long long*>(ptr), scalars,
        kstar, exact);
    return cudaGetLastError() == cudaSuccess ? VERKV_OK : VERKV_ECUDA;
}
