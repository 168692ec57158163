// KVFetch on the GPU: sketch scores, the bounded-shrinkage fixed point, the Bernstein
// certificate, gains, ranking, k*, the union fetch from pinned host memory and the weighted
// attention.  Paper: "Verify Before You Fetch: Reliable KV Cache Compression for LLM Inference",
// Algorithm 2 / Sec. 4.2 (Definition 2 / eq. (5), Lemma 1 / eq. (7), eqs. (9)-(10), Theorem 2),
// Appendix A.1 (sketch), Appendix A.3.2 (decide / fetch / attention kernels: prior art).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <type_traits>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "async.cuh"
#include "umma.cuh"

namespace cg = cooperative_groups;

namespace verkv {

namespace {

constexpr int kMaxBatch = 32;
constexpr int kTile = 128;      // token positions per score block (= 2-bit sketch group)
constexpr int kSelWidth = 4096; // candidates ranked on chip per row

struct Views {
    SlotView v[kMaxBatch];
};

struct DecodeArgs {
    uint32_t* ebits;  // [B Hq][ws_n/32 + 1] per query row: tokens of L_g[:k*] \ S (set by the decision kernels)
    float* om;        // [B Hq][ws_n] weight factor of each resident slot (set by the scoring and decision kernels)
    int* err;         // mapped host word, set when a bounded device-side wait gives up
    int* done;        // [B Hkv] attention blocks finished per KV head (the last one merges; left at 0)
    int32_t* hrows;   // [B Hkv] rows read over the host link (zeroed by the scoring kernel of the call)
    // speculative prefetch (see prefetch_kernel): rows copied ahead, their maps and counters
    unsigned char* pf_buf;
    int32_t* pf_of;
    int32_t* pf_tok;
    int32_t* pf_cnt;
    int32_t* pf_used;
    unsigned long long* dprog;
    // call timeline (null: off): device times of the first CTA start ([0] scoring, [1] decision after
    // its dependency wait, [2] prefetch, [3] attention after its wait) and of the last CTA end ([8]
    // decision, [9] prefetch binning, [10] prefetch, [11] attention), in globaltimer nanoseconds
    unsigned long long* tline;
    int pf_cap;       // rows per (sequence, KV head); 0: the prefetch is off for this call
    int Hkv, Hq, G, ws_n, ws_npow2, gen, nsplit;
    int binary;       // 1: binary shrinkage coefficients (lambda in {1, r}), 0: the clipped fixed point
    float eps_f;
    double eps, ldelta;
    ff eps_ff, ld_ff;   // eps and log(2/delta) as float-float
    float inv_sqrt_d_f;
    ff inv_sqrt_d;
};

__device__ __forceinline__ int row_of(int b, int hq, int Hq) { return b * Hq + hq; }

// Call timeline entry k: the earliest (first) or the latest (!first) time any CTA reached it.
__device__ __forceinline__ void tline_stamp(unsigned long long* t, int k, bool first)
{
    if (t) {
        const unsigned long long v = global_ns();
        if (first) atomicMin(t + k, v);
        else atomicMax(t + k, v);
    }
}

// K/V row elements (bf16 or fp32) to fp32: eight channels from 16 (or 32) bytes, or a pair.
template <typename T> struct RowCvt;
template <> struct RowCvt<__nv_bfloat16> {
    // 8 channels from 16 bytes
    static __device__ __forceinline__ void load8(const void* p, float* o)
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            o[2 * k] = f.x;
            o[2 * k + 1] = f.y;
        }
    }
    static __device__ __forceinline__ float2 load2(const void* p)
    {
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    }
};
template <> struct RowCvt<float> {
    static __device__ __forceinline__ void load8(const void* p, float* o)
    {
        const float4 x = reinterpret_cast<const float4*>(p)[0], y = reinterpret_cast<const float4*>(p)[1];
        o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
        o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
    }
    static __device__ __forceinline__ float2 load2(const void* p) { return *reinterpret_cast<const float2*>(p); }
};


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
    s.m_tag = 0;
    s.n_h = views.v[b].counts[kv * 4 + 0] + views.v[b].n_tail;   // appended tokens are H
    s.n_l = views.v[b].counts[kv * 4 + 1];
    s.b_arg = -1;
    rows[row] = s;
}

// --------------------------------------------------------------------------------------------
// D1: sketch logits <q, k^_i>/sqrt(d) of the tokens of L, as float-float.  The query side is split so
// that the bulk of each dot product is an exact sum of integer multiples of a power of two:
//   int8:  q = 2^(E-10) P1 + 2^(E-21) P2 + 2^(E-32) P3 + r (|q| < 2^E, |r| <= 2^(E-33)) with integer
//          pieces |P| <= 1024, exact in fp16, as are the codes |c| <= 127; every sum over the 128
//          channels of P c is an integer below 2^24, so the tensor core's fp32 accumulation of those
//          products is exact.  One M = 128 tokens x N = (3 pieces x G heads, padded) x K = 128 MMA per
//          tile of 128 tokens, accumulated in tensor memory.
//   2-bit: kappa_j = q_j * scale_gj (exact two-product), split on the grid 2^(E-17) of the group;
//          codes are 0..3 and 32 channels, so the grid part is exact as well.
// --------------------------------------------------------------------------------------------
__device__ __forceinline__ ff combine3(float s1, float s2, float s3)
{
    ff t = two_sum(s1, s2);
    return fast_two_sum(t.hi, __fadd_rn(t.lo, s3));
}

// Exact logits of the tokens of H (resident keys), by H index: U tiles of kTile / (8 G) tokens each,
// tiles t0, t0 + stride, ..., 8 threads per (token, query head), 16 channels each (float-float
// partial sums combined over the 8 lanes).  The resident slots and key rows of all U tiles are loaded
// before any is used.  Also sets the weight factor of each token's resident slot to 1 for every query
// head.
template <typename T, int G, int U>
__device__ __forceinline__ void score_h_tiles(const Views& views, const float* __restrict__ q, const DecodeArgs& a,
                                              RowState* __restrict__ rows, float2* __restrict__ th, int t0, int stride)
{
    constexpr int TPB = kTile / (8 * G);
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int nh0 = V.counts[kv * 4 + 0], nh = nh0 + V.n_tail;   // H of the compress, then appended tokens
    const int t = threadIdx.x;
    const int part = t & 7, g = (t >> 3) % G, tk = t / (8 * G);
    const int row = row_of(b, kv * G + g, a.Hq);
    int hk[U], slot[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        hk[u] = (t0 + u * stride) * TPB + tk;
        slot[u] = hk[u] < nh0 ? V.hslot[(int64_t)kv * n + hk[u]] : V.counts[kv * 4 + 3] + (hk[u] - nh0);
    }
    float kk[U][16];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (hk[u] < nh) {
            const T* key = reinterpret_cast<const T*>(V.kvres) + (V.res_off[kv] + slot[u]) * 2 * kHeadDim + part * 16;
            RowCvt<T>::load8(key, kk[u]);
            RowCvt<T>::load8(key + 8, kk[u] + 8);
        }
    }
    float qq[16];
    {
        const float* qr = q + (int64_t)row * kHeadDim + part * 16;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            const float4 x = reinterpret_cast<const float4*>(qr)[c4];
            qq[4 * c4] = x.x;
            qq[4 * c4 + 1] = x.y;
            qq[4 * c4 + 2] = x.z;
            qq[4 * c4 + 3] = x.w;
        }
    }
    float mloc = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool live = hk[u] < nh;
        ff s = {0.f, 0.f};
        if (live) {
            float hi = 0.f, lo = 0.f;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const ff p = two_prod(qq[c], kk[u][c]);
                const ff w = two_sum(hi, p.hi);
                hi = w.hi;
                lo = __fadd_rn(lo, __fadd_rn(w.lo, p.lo));
            }
            s = fast_two_sum(hi, lo);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) s = ff_add(s, shfl_xor_ff(s, o));
        if (live && part == 0) {
            const ff x = ff_mul(s, a.inv_sqrt_d);
            th[(int64_t)row * a.ws_n + hk[u]] = make_float2(x.hi, x.lo);
            a.om[(int64_t)row * a.ws_n + slot[u]] = 1.0f;   // H: weight factor 1
            mloc = fmaxf(mloc, x.hi);
        }
    }
    // max per query head: lanes of head g are the 8-lane groups with the same g in the warp
    for (int o = 8 * G; o < 32; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
    if ((threadIdx.x & 31) < 8 * G && part == 0 && mloc > -INFINITY)
        atomicMax(&rows[row].m_tag, tag_max((unsigned)a.gen, mloc));
}

// kHTilesPerBlock consecutive H tiles per block, so that the L and H blocks of a scoring launch fit in
// one wave of resident blocks.
constexpr int kHTilesPerBlock = 4;

template <typename T, int G>
__device__ __forceinline__ void score_h_tile(const Views& views, const float* __restrict__ q, const DecodeArgs& a,
                                             RowState* __restrict__ rows, float2* __restrict__ th, int block)
{
    // two tiles at a time: the blocks of this path share the register budget of the L-tile blocks
    for (int t = 0; t < kHTilesPerBlock; t += 2)
        score_h_tiles<T, G, 2>(views, q, a, rows, th, block * kHTilesPerBlock + t, 1);
}

// 2-bit sketch tile: GPB sketch groups (of kTile tokens) per block; warp w scores group w, each
// lane four tokens of it, so every shared-memory load of the query split (four channels at a
// time) serves four tokens.
constexpr int kGroupsPerBlock = kTile / 32;

template <typename T, int G>
__global__ void __launch_bounds__(kTile) score_2bit_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                           RowState* __restrict__ rows, float2* __restrict__ tl,
                                                           float2* __restrict__ th, int n_ltiles)
{
    pdl_trigger();   // the decision kernel may start its independent prologue
    if (threadIdx.x == 0) tline_stamp(a.tline, 0, true);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.hrows[blockIdx.y] = 0;   // host rows of this call (attention)
        a.pf_cnt[blockIdx.y] = 0;   // rows the prefetch claims, and of them the attention reads
        a.pf_used[blockIdx.y] = 0;
        if (blockIdx.y == 0) *a.dprog = (unsigned long long)(unsigned)a.gen << 32;   // no row decided yet
    }
    if ((int)blockIdx.x >= n_ltiles) {
        score_h_tile<T, G>(views, q, a, rows, th, blockIdx.x - n_ltiles);
        return;
    }
    constexpr int NP = kHeadDim / 8, KEPT = kHeadDim / 4, GPB = kGroupsPerBlock, TPT = kTile / 32;
    __shared__ __align__(16) float k1[GPB][G][KEPT];
    __shared__ __align__(16) float rho[GPB][G][KEPT];
    __shared__ ff zsum[GPB][G];
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int ngroups = (n + kTile - 1) / kTile;
    const int grp0 = blockIdx.x * GPB;
    if (grp0 >= ngroups) return;  // a shorter sequence of the batch
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float* qb = q + ((int64_t)b * a.Hq + kv * G) * kHeadDim;
    // per (group, head): kappa_j = q_ch * scale, Z = sum_j q_ch * zero, grid split of kappa.  Warp w
    // takes group w, lane j kept channel j; every load is issued before the arithmetic.
    {
        const int gi = warp, grp = grp0 + gi;
        if (grp < ngroups) {
            const int j = lane;
            const int64_t pi = ((int64_t)kv * ngroups + grp) * KEPT + j;
            const float z = __half2float(V.zero2[pi]), sc = __half2float(V.scale2[pi]);
            const int p = V.pairs[kv * NP + (j % NP)];
            const int ch = j < NP ? p : p + kHeadDim / 2;
            float qc[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) qc[gg] = qb[gg * kHeadDim + ch];
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const ff kap = two_prod(qc[gg], sc);
                const ff zz = warp_sum_ff(two_prod(qc[gg], z));
                const float mx = warp_max(fabsf(kap.hi));
                int E;
                frexpf(mx, &E);
                const float K1 = ldexpf(rintf(ldexpf(kap.hi, 17 - E)), E - 17);
                k1[gi][gg][j] = K1;
                rho[gi][gg][j] = __fadd_rn(__fsub_rn(kap.hi, K1), kap.lo);
                if (j == 0) zsum[gi][gg] = zz;
            }
        }
    }
    __syncthreads();
    const int gi = warp, grp = grp0 + gi;
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    if (grp < ngroups) {
        int li[TPT];
        uint64_t w[TPT];
#pragma unroll
        for (int t = 0; t < TPT; ++t) {
            const int i = grp * kTile + lane + 32 * t;
            li[t] = i < n ? V.lpos[(int64_t)kv * n + i] : -1;   // < 0: not in L
            w[t] = li[t] >= 0 ? V.codes2[(int64_t)kv * n + i] : 0ull;
        }
        float s1[TPT][G], s2[TPT][G];
#pragma unroll
        for (int t = 0; t < TPT; ++t)
#pragma unroll
            for (int g = 0; g < G; ++g) s1[t][g] = s2[t][g] = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < KEPT; j4 += 4) {
            float cf[TPT][4];
#pragma unroll
            for (int t = 0; t < TPT; ++t)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) cf[t][jj] = (float)((unsigned)(w[t] >> (2 * (j4 + jj))) & 3u);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 K = *reinterpret_cast<const float4*>(&k1[gi][g][j4]);
                const float4 R = *reinterpret_cast<const float4*>(&rho[gi][g][j4]);
                const float kq[4] = {K.x, K.y, K.z, K.w}, rq[4] = {R.x, R.y, R.z, R.w};
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                    for (int t = 0; t < TPT; ++t) {
                        s1[t][g] = __fmaf_rn(kq[jj], cf[t][jj], s1[t][g]);
                        s2[t][g] = __fmaf_rn(rq[jj], cf[t][jj], s2[t][g]);
                    }
            }
        }
#pragma unroll
        for (int t = 0; t < TPT; ++t) {
            if (li[t] < 0) continue;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                ff x = ff_add(zsum[gi][g], two_sum(s1[t][g], s2[t][g]));
                x = ff_mul(x, a.inv_sqrt_d);
                const int row = row_of(b, kv * G + g, a.Hq);
                tl[(int64_t)row * a.ws_n + li[t]] = make_float2(x.hi, x.lo);
                mloc[g] = fmaxf(mloc[g], x.hi);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m = warp_max(mloc[g]);
        if (lane == 0 && m > -INFINITY) atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_tag, tag_max((unsigned)a.gen, m));
    }
}

// Int8 sketch tiles on the tensor cores.  A CTA scores a contiguous range of 128-token tiles of one
// (sequence, KV head): A = the tile's codes as fp16 (128 tokens x 128 channels, K-major, 128-byte
// swizzle; two stages), B = the query pieces (N rows: piece k of head g in row 3 g + k), D = two
// tensor-memory accumulators of N fp32 columns.  The codes of the next two tiles (and each thread's
// L position and scale) are in flight in registers while the current tile is converted and its MMAs
// run next to the epilogue of the previous tile; warp w holds tokens 32 w .. 32 w + 31 of a tile
// (its tensor-memory lane quarter) and finishes one token per thread.  The grid is one wave of
// kInt8CtasPerSm CTAs per multiprocessor; after its tiles, each CTA also takes a share of the exact
// logits of the KV head's H tokens.
template <int G>
struct Int8Mma {
    static constexpr int NP = (3 * G + 15) / 16 * 16;           // B rows, padded to the MMA's N step
    static constexpr int COLS = 2 * NP < 32 ? 32 : 2 * NP;      // tensor-memory columns (two accumulators)
    static constexpr int ABytes = 128 * kHeadDim * 2;           // one fp16 code tile (32 KiB)
    static constexpr int BBytes = NP * kHeadDim * 2;
    static constexpr size_t Smem = 2 * (size_t)ABytes + BBytes + 1024;   // + alignment slack
};
constexpr int kInt8CtasPerSm = 3;

// Four int8 codes (one 32-bit word) to four exact fp16 values: the sign bits are flipped (c + 128),
// each byte is placed under the fp16 exponent of 1024 (1024 + c + 128, exact) and 1152 subtracted.
__device__ __forceinline__ uint2 codes4_to_f16(uint32_t w)
{
    const uint32_t x = w ^ 0x80808080u;
    uint32_t lo = __byte_perm(x, 0x64646464u, 0x4140), hi = __byte_perm(x, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480u), __ushort_as_half((unsigned short)0x6480u));
    __half2 l2 = __hsub2(*reinterpret_cast<__half2*>(&lo), bias), h2 = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
    return make_uint2(*reinterpret_cast<uint32_t*>(&l2), *reinterpret_cast<uint32_t*>(&h2));
}

template <typename T, int G>
__device__ __forceinline__ void score_int8_ltiles(const Views& views, const float* __restrict__ q, const DecodeArgs& a,
                                                  RowState* __restrict__ rows, float2* __restrict__ tl, int b, int kv,
                                                  int t0, int nt)
{
    using P = Int8Mma<G>;
    extern __shared__ unsigned char dsm_raw[];
    __shared__ __align__(8) unsigned long long bar[2];
    __shared__ unsigned tbase;
    __shared__ float red[32];
    __shared__ int qexp[G];
    unsigned char* dsm = dsm_raw + ((1024u - (umma_smem_u32(dsm_raw) & 1023u)) & 1023u);
    unsigned char* sA = dsm;
    unsigned char* sB = dsm + 2 * P::ABytes;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // B: the pieces of the G query rows (thread c owns channel c), rows past 3 G zero
    const float* qg = q + ((int64_t)b * a.Hq + kv * G) * kHeadDim;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float v = qg[g * kHeadDim + tid];
        const float mx = block_max(fabsf(v), red);
        int E;
        frexpf(mx, &E);   // mx < 2^E (E = 0 for a zero query)
        const float p1 = rintf(ldexpf(v, 10 - E));
        const float r1 = __fsub_rn(v, ldexpf(p1, E - 10));
        const float p2 = rintf(ldexpf(r1, 21 - E));
        const float r2 = __fsub_rn(r1, ldexpf(p2, E - 21));
        const float p3 = rintf(ldexpf(r2, 32 - E));
        *reinterpret_cast<__half*>(sB + umma_sw128_offset(3 * g + 0, tid, P::NP)) = __float2half_rn(p1);
        *reinterpret_cast<__half*>(sB + umma_sw128_offset(3 * g + 1, tid, P::NP)) = __float2half_rn(p2);
        *reinterpret_cast<__half*>(sB + umma_sw128_offset(3 * g + 2, tid, P::NP)) = __float2half_rn(p3);
        if (tid == 0) qexp[g] = E;
    }
    for (int r = 3 * G; r < P::NP; ++r) *reinterpret_cast<__half*>(sB + umma_sw128_offset(r, tid, P::NP)) = __float2half_rn(0.f);

    // codes of tile i into registers: lane l of warp w reads the 16-byte chunk l % 8 of tokens
    // 32 w + 4 j + l / 8 (j = 0..7): each load instruction of the warp covers 512 contiguous bytes.
    // With them, the L position and scale of this thread's own token of the tile (its epilogue row).
    const int8_t* codes = V.codes8 + (int64_t)kv * n * kHeadDim;
    auto load = [&](int i, uint4 (&buf)[8], int& li, float& sc) {
        const int tok0 = (t0 + i) * 128 + 32 * warp + (lane >> 3);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int tok = tok0 + 4 * j;
            buf[j] = tok < n ? __ldg(reinterpret_cast<const uint4*>(codes + (int64_t)tok * kHeadDim) + (lane & 7))
                             : make_uint4(0u, 0u, 0u, 0u);
        }
        const int tok = (t0 + i) * 128 + 32 * warp + lane;
        li = tok < n ? __ldg(V.lpos + (int64_t)kv * n + tok) : -1;   // < 0: not in L
        sc = tok < n ? __ldg(V.scale8 + (int64_t)kv * n + tok) : 0.f;
    };
    auto store = [&](int i, const uint4 (&buf)[8]) {
        unsigned char* dst = sA + (i & 1) * P::ABytes;
        const int k0 = 16 * (lane & 7);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = 32 * warp + 4 * j + (lane >> 3);
            const uint2 c0 = codes4_to_f16(buf[j].x), c1 = codes4_to_f16(buf[j].y), c2 = codes4_to_f16(buf[j].z),
                        c3 = codes4_to_f16(buf[j].w);
            *reinterpret_cast<uint4*>(dst + umma_sw128_offset(row, k0, 128)) = make_uint4(c0.x, c0.y, c1.x, c1.y);
            *reinterpret_cast<uint4*>(dst + umma_sw128_offset(row, k0 + 8, 128)) = make_uint4(c2.x, c2.y, c3.x, c3.y);
        }
    };
    // two tiles in flight: register set 0 holds even tiles, set 1 odd tiles
    uint4 buf0[8], buf1[8];
    int li0 = -1, li1 = -1, li_ep = -1;
    float sc0 = 0.f, sc1 = 0.f, sc_ep = 0.f;
    load(0, buf0, li0, sc0);
    if (nt > 1) load(1, buf1, li1, sc1);
    if (warp == 0) umma_alloc(&tbase, P::COLS);
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    umma_fence_before();
    __syncthreads();
    umma_fence_after();
    const unsigned tmem = tbase;
    constexpr unsigned idesc = umma_idesc_f16_f32(128, P::NP);
    int E[G];
#pragma unroll
    for (int g = 0; g < G; ++g) E[g] = qexp[g];
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    bool bad = false;
    // step i converts tile i (from its register set, which then starts loading tile i + 2) and issues
    // its MMAs, then finishes tile i - 1, whose MMAs ran meanwhile
    auto step = [&](int i, uint4 (&buf)[8], int& li, float& sc) {
        int li_t = -1;
        float sc_t = 0.f;
        if (i < nt) {
            li_t = li;
            sc_t = sc;
            store(i, buf);   // stage i % 2: the MMAs of tile i - 2 that read it are complete (waited at i - 1)
            if (i + 2 < nt) load(i + 2, buf, li, sc);
            fence_proxy_async_smem();   // the fp16 tiles (generic stores) -> tensor core
            umma_fence_before();
            __syncthreads();   // tile i is in shared memory; accumulator i % 2 was read back at i - 1
            if (tid == 0) {
                umma_fence_after();
                const unsigned d = tmem + (unsigned)((i & 1) * P::NP);
                const unsigned ab = umma_smem_u32(sA + (i & 1) * P::ABytes), bb = umma_smem_u32(sB);
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 16; ++ks)
                    umma_mma(d, umma_desc_sw128(ab + umma_kstep_offset(ks, 128)),
                             umma_desc_sw128(bb + umma_kstep_offset(ks, P::NP)), idesc, ks > 0);
                umma_commit(&bar[i & 1]);
            }
        }
        if (i >= 1 && i <= nt) {
            const int e = i - 1;
            if (!mbar_wait(&bar[e & 1], (unsigned)((e >> 1) & 1), kWaitLimit)) bad = true;
            umma_fence_after();
            float acc[P::NP];
            const unsigned ta = tmem + ((unsigned)(32 * warp) << 16) + (unsigned)((e & 1) * P::NP);
#pragma unroll
            for (int c = 0; c < P::NP; c += 16) umma_ld16(ta + c, *reinterpret_cast<float(*)[16]>(acc + c));
            umma_fence_before();
            if (li_ep >= 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    ff x = combine3(ldexpf(acc[3 * g], E[g] - 10), ldexpf(acc[3 * g + 1], E[g] - 21),
                                    ldexpf(acc[3 * g + 2], E[g] - 32));
                    x = ff_mul(ff_mul_f(x, sc_ep), a.inv_sqrt_d);
                    const int row = row_of(b, kv * G + g, a.Hq);
                    tl[(int64_t)row * a.ws_n + li_ep] = make_float2(x.hi, x.lo);
                    mloc[g] = fmaxf(mloc[g], x.hi);
                }
            }
        }
        li_ep = li_t;
        sc_ep = sc_t;
    };
    for (int i = 0; i <= nt; i += 2) {
        step(i, buf0, li0, sc0);
        step(i + 1, buf1, li1, sc1);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m = warp_max(mloc[g]);
        if (lane == 0 && m > -INFINITY) atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_tag, tag_max((unsigned)a.gen, m));
    }
    if (bad) *(volatile int*)a.err = 1;
    __syncthreads();
    if (warp == 0) {
        umma_fence_after();
        umma_dealloc(tmem, P::COLS);
    }
}

template <typename T, int G>
__global__ void __launch_bounds__(kTile, kInt8CtasPerSm) score_int8_kernel(Views views, const float* __restrict__ q,
                                                                            DecodeArgs a, RowState* __restrict__ rows,
                                                                            float2* __restrict__ tl,
                                                                            float2* __restrict__ th, int n_lchunks)
{
    pdl_trigger();   // the decision kernel may start its independent prologue
    if (threadIdx.x == 0) tline_stamp(a.tline, 0, true);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.hrows[blockIdx.y] = 0;   // host rows of this call (attention)
        a.pf_cnt[blockIdx.y] = 0;   // rows the prefetch claims, and of them the attention reads
        a.pf_used[blockIdx.y] = 0;
        if (blockIdx.y == 0) *a.dprog = (unsigned long long)(unsigned)a.gen << 32;   // no row decided yet
    }
    const int b = blockIdx.y / a.Hkv, kv = blockIdx.y % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int ntiles = (n + 127) / 128;
    const int per = (ntiles + n_lchunks - 1) / n_lchunks;
    const int t0 = blockIdx.x * per, nt = min(ntiles, t0 + per) - t0;
    if (nt > 0) score_int8_ltiles<T, G>(views, q, a, rows, tl, b, kv, t0, nt);
    // the exact logits of the KV head's H tokens, shared out over its CTAs
    constexpr int TPB = kTile / (8 * G);
    const int nh_tiles = (V.counts[kv * 4 + 0] + V.n_tail + TPB - 1) / TPB;
    for (int ht = blockIdx.x; ht < nh_tiles; ht += kHTilesPerBlock * gridDim.x)
        score_h_tiles<T, G, kHTilesPerBlock>(views, q, a, rows, th, ht, gridDim.x);
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

// --------------------------------------------------------------------------------------------
// Shortlist and exact certificate weights (App. A.1; launched only when enabled), two kernels.
// shortlist_keys_kernel: blocks y < ny_keys of a (sequence, KV head) each take a slice of L.  The key
// of every entry -- the order-preserving bits of its largest sketch logit over the head's G query
// rows, ascending = descending score; ~0u for sampled entries, which are no candidates -- goes into a
// scratch row (the full-row ranking's key buffer, idle at this point of a call) and into the KV
// head's first-level histogram (top 12 bits) in global memory.  Blocks y >= ny_keys replace the
// sketch logits of the sampled tokens (their keys are resident) by exact ones.
// shortlist_select_kernel: one block per (sequence, KV head) finishes the radix select of the k-th
// key (levels of 12 and 8 more bits over the scratch), takes the tokens below it and the first at it
// in L order (ties by lower L index, i.e. token order), reads their keys from the pinned host cache,
// scores them exactly and clears the histogram for the next call.  Every exact logit also raises its
// row's maximum.  The two kinds of blocks of the first kernel touch disjoint entries of the logits.
// --------------------------------------------------------------------------------------------
constexpr int kSlThreads = 512;
constexpr int kSlBins = kShortlistBins;

// Exact float-float logits <q_g, k>/sqrt(d) of one key row for the G query rows q0 + g d: the key is
// read 16 bytes at a time (once for all heads), every product is a two-product, the sums carry their
// rounding errors.
template <typename T, int G>
__device__ __forceinline__ void exact_logits_row(const float* __restrict__ q0, const T* key, ff inv_sqrt_d,
                                                 ff (&out)[G])
{
    float hi[G], lo[G];
#pragma unroll
    for (int g = 0; g < G; ++g) hi[g] = lo[g] = 0.f;
    const unsigned char* kb = reinterpret_cast<const unsigned char*>(key);
    // bf16 rows: all 16 words of the key in flight at once (one round trip when it is host memory)
    constexpr bool kPre = std::is_same<T, __nv_bfloat16>::value;
    uint4 kr[kPre ? kHeadDim / 8 : 1];
    if constexpr (kPre) {
#pragma unroll
        for (int j = 0; j < kHeadDim / 8; ++j) kr[j] = reinterpret_cast<const uint4*>(kb)[j];
    }
#pragma unroll 4
    for (int c8 = 0; c8 < kHeadDim; c8 += 8) {
        float kk[8];
        if constexpr (kPre)
            RowCvt<T>::load8(&kr[c8 / 8], kk);
        else
            RowCvt<T>::load8(kb + c8 * (int)sizeof(T), kk);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float4 qa = *reinterpret_cast<const float4*>(q0 + g * kHeadDim + c8);
            const float4 qb = *reinterpret_cast<const float4*>(q0 + g * kHeadDim + c8 + 4);
            const float qq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const ff p = two_prod(qq[c], kk[c]);
                const ff t = two_sum(hi[g], p.hi);
                hi[g] = t.hi;
                lo[g] = __fadd_rn(lo[g], __fadd_rn(t.lo, p.lo));
            }
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) out[g] = ff_mul(fast_two_sum(hi[g], lo[g]), inv_sqrt_d);
}

// The same logits with one key row spread over four adjacent lanes: lane part p (0..3) sums channels
// [32 p, 32 p + 32) and the four float-float partial sums are combined by error-free additions, so
// every lane of the group ends with the same result.  Every lane of the warp must call it; a lane with
// no row passes key = nullptr and reads nothing.
template <typename T, int G>
__device__ __forceinline__ void exact_logits_quad(const float* __restrict__ q0, const T* key, int part,
                                                  ff inv_sqrt_d, ff (&out)[G])
{
    constexpr int kQ = kHeadDim / 4;   // channels of one lane
    float hi[G], lo[G];
#pragma unroll
    for (int g = 0; g < G; ++g) hi[g] = lo[g] = 0.f;
    if (key != nullptr) {
        const unsigned char* kb = reinterpret_cast<const unsigned char*>(key + part * kQ);
        constexpr int kWords = kQ * (int)sizeof(T) / 16;
        uint4 kr[kWords];   // the lane's part of the row in flight at once
#pragma unroll
        for (int j = 0; j < kWords; ++j) kr[j] = reinterpret_cast<const uint4*>(kb)[j];
#pragma unroll
        for (int c8 = 0; c8 < kQ; c8 += 8) {
            float kk[8];
            RowCvt<T>::load8(reinterpret_cast<const unsigned char*>(kr) + c8 * (int)sizeof(T), kk);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float* qg = q0 + g * kHeadDim + part * kQ + c8;
                const float4 qa = *reinterpret_cast<const float4*>(qg);
                const float4 qb = *reinterpret_cast<const float4*>(qg + 4);
                const float qq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const ff p = two_prod(qq[c], kk[c]);
                    const ff t = two_sum(hi[g], p.hi);
                    hi[g] = t.hi;
                    lo[g] = __fadd_rn(lo[g], __fadd_rn(t.lo, p.lo));
                }
            }
        }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float oh = __shfl_xor_sync(0xffffffffu, hi[g], o), ol = __shfl_xor_sync(0xffffffffu, lo[g], o);
            const ff t = two_sum(hi[g], oh);
            hi[g] = t.hi;
            lo[g] = __fadd_rn(__fadd_rn(lo[g], ol), t.lo);
        }
#pragma unroll
    for (int g = 0; g < G; ++g) out[g] = ff_mul(fast_two_sum(hi[g], lo[g]), inv_sqrt_d);
}

// 32-bit words of a KV head's scratch key row (a multiple of four)
__device__ __forceinline__ int64_t shortlist_stride(const DecodeArgs& a) { return 2 * (int64_t)max(a.ws_npow2, 2); }

__device__ __forceinline__ unsigned score_key(float s)   // ascending key = descending score
{
    return ~((unsigned)float_to_ordered(s) ^ 0x80000000u);
}

template <typename T, int G>
__global__ void __launch_bounds__(kSlThreads) shortlist_keys_kernel(Views views, const float* __restrict__ q,
                                                                   DecodeArgs a, RowState* rows, float2* tl,
                                                                   unsigned* __restrict__ skeys,
                                                                   unsigned* __restrict__ ghist, int ny_keys)
{
    const int unit = blockIdx.x, b = unit / a.Hkv, kv = unit % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int nl = V.counts[kv * 4 + 1];
    const int row0 = row_of(b, kv * G, a.Hq);
    const int tid = threadIdx.x, lane = tid & 31;
    if ((int)blockIdx.y >= ny_keys) {
        // sampled tokens: resident slot rs -> token -> L index (H tokens have none)
        float mloc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
        const int m_res = V.counts[kv * 4 + 3];
        const int rs = ((int)blockIdx.y - ny_keys) * (kSlThreads / 4) + tid / 4, part = tid & 3;
        int li = -1;
        const T* key = nullptr;
        if (rs < m_res) {
            const int tok = V.rtok[(int64_t)kv * n + rs];
            li = V.lpos[(int64_t)kv * n + tok];
            if (li >= 0) key = reinterpret_cast<const T*>(V.kvres) + (V.res_off[kv] + rs) * 2 * kHeadDim;
        }
        ff x[G];
        exact_logits_quad<T, G>(q + (int64_t)row0 * kHeadDim, key, part, a.inv_sqrt_d, x);
        if (key != nullptr) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                if (part == 0) tl[(int64_t)(row0 + g) * a.ws_n + li] = make_float2(x[g].hi, x[g].lo);
                mloc[g] = fmaxf(mloc[g], x[g].hi);
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float m = warp_max(mloc[g]);
            if (lane == 0 && m > -INFINITY) atomicMax(&rows[row0 + g].m_tag, tag_max((unsigned)a.gen, m));
        }
        return;
    }
    __shared__ unsigned hist[kSlBins];
    for (int i = tid; i < kSlBins; i += kSlThreads) hist[i] = 0u;
    __syncthreads();
    unsigned* sk = skeys + unit * shortlist_stride(a);
    const int nl4 = (nl + 3) / 4;
    const int per = (nl4 + ny_keys - 1) / ny_keys;
    const int a0 = min(nl4, (int)blockIdx.y * per), a1 = min(nl4, a0 + per);
    int nc = 0;
    for (int i4 = a0 + tid; i4 < a1; i4 += kSlThreads) {
        int sl4[4];
        float2 t4[4][G];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int li = 4 * i4 + u;
            sl4[u] = li < nl ? V.lslot[(int64_t)kv * n + li] : 0;
#pragma unroll
            for (int g = 0; g < G; ++g)
                t4[u][g] = li < nl ? tl[(int64_t)(row0 + g) * a.ws_n + li] : make_float2(0.f, 0.f);
        }
        unsigned kk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float sc = -INFINITY;
#pragma unroll
            for (int g = 0; g < G; ++g) sc = fmaxf(sc, t4[u][g].x);
            const bool cand = 4 * i4 + u < nl && sl4[u] < 0;
            kk[u] = cand ? score_key(sc) : ~0u;
            if (cand) {
                ++nc;
                atomicAdd(&hist[kk[u] >> 20], 1u);
            }
        }
        reinterpret_cast<uint4*>(sk)[i4] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
    }
    __syncthreads();
    unsigned* gh = ghist + (int64_t)unit * (kSlBins + 1);   // bins, then the candidate count
    for (int i = tid; i < kSlBins; i += kSlThreads)
        if (hist[i]) atomicAdd(&gh[i], hist[i]);
    nc = __reduce_add_sync(0xffffffffu, (unsigned)nc);
    if (lane == 0 && nc > 0) atomicAdd(&gh[kSlBins], (unsigned)nc);
}

// Calls f(key, L index) for every scratch key of a row, eight 16-byte words per thread in flight.
template <typename F>
__device__ __forceinline__ void for_each_key(const uint4* __restrict__ sk4, int nl4, int tid, F&& f)
{
    constexpr int kB = 8;
    for (int base = 0; base < nl4; base += kB * kSlThreads) {
        uint4 kq[kB];
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int i4 = base + j * kSlThreads + tid;
            kq[j] = i4 < nl4 ? sk4[i4] : make_uint4(~0u, ~0u, ~0u, ~0u);
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
            const int li = 4 * (base + j * kSlThreads + tid);
            f(kq[j].x, li);
            f(kq[j].y, li + 1);
            f(kq[j].z, li + 2);
            f(kq[j].w, li + 3);
        }
    }
}

constexpr int kSlCand = 2048;   // keys of the threshold's first-level bin ranked in shared memory

template <typename T, int G>
__global__ void __launch_bounds__(kSlThreads) shortlist_select_kernel(Views views, const float* __restrict__ q,
                                                                     DecodeArgs a, RowState* rows, float2* tl,
                                                                     int k_short, int32_t* __restrict__ slist,
                                                                     int32_t* __restrict__ scount,
                                                                     const unsigned* __restrict__ skeys,
                                                                     unsigned* __restrict__ ghist)
{
    const int unit = blockIdx.x, b = unit / a.Hkv, kv = unit % a.Hkv;
    const SlotView& V = views.v[b];
    const int n = V.n;
    const int nl = V.counts[kv * 4 + 1];
    const int row0 = row_of(b, kv * G, a.Hq);
    const int tid = threadIdx.x;
    __shared__ unsigned hist[kSlBins];
    __shared__ int s_scan[32];
    __shared__ unsigned s_prefix;
    __shared__ int s_need, s_count, s_at_thr, s_ncand;
    __shared__ int s_sel[kMaxShortlist];
    __shared__ uint2 s_cand[kSlCand];
    unsigned* gh = ghist + (int64_t)unit * (kSlBins + 1);
    // the first-level histogram, every word in flight at once
    {
        unsigned hv[kSlBins / kSlThreads];
#pragma unroll
        for (int j = 0; j < kSlBins / kSlThreads; ++j) hv[j] = __ldcg(gh + tid + j * kSlThreads);
#pragma unroll
        for (int j = 0; j < kSlBins / kSlThreads; ++j) hist[tid + j * kSlThreads] = hv[j];
    }
    const int ntot = (int)__ldcg(gh + kSlBins);
    const int k = min(k_short, ntot);
    const int nl4 = (nl + 3) / 4;
    const uint4* sk4 = reinterpret_cast<const uint4*>(skeys + unit * shortlist_stride(a));
    if (tid == 0) {
        s_prefix = 0u;
        s_need = k;
        s_count = 0;
        s_at_thr = 0;
        s_ncand = 0;
    }
    __syncthreads();
    // the histogram is read: leave it clear for the next call
#pragma unroll
    for (int j = 0; j < kSlBins / kSlThreads; ++j) gh[tid + j * kSlThreads] = 0u;
    if (tid == 0) gh[kSlBins] = 0u;
    // radix select of the k-th key.  A level stops the search once every key of the digit it found
    // is taken; after the first level, a bin of at most kSlCand keys is ranked in shared memory.
    unsigned lowmask = 0u;
    bool cand = false;
    for (int lev = 0; lev < 3 && k > 0 && k < ntot; ++lev) {
        const int sh = lev == 0 ? 20 : lev == 1 ? 8 : 0, wd = lev < 2 ? 12 : 8, nb = 1 << wd;   // 12, 12, 8 bits
        const unsigned prefix = s_prefix;
        const int need = s_need;
        if (lev > 0) {   // level 0 comes from the keys kernel
            for (int i = tid; i < nb; i += kSlThreads) hist[i] = 0u;
            __syncthreads();
            for_each_key(sk4, nl4, tid, [&](unsigned key, int) {
                if (key != ~0u && (key >> (sh + wd)) == (prefix >> (sh + wd)))
                    atomicAdd(&hist[(key >> sh) & (nb - 1)], 1u);
            });
            __syncthreads();
        }
        // the digit holding the need-th key: bins of this thread, then a block scan of their sums
        const int per = (nb + kSlThreads - 1) / kSlThreads;
        const int d0 = min(nb, tid * per), d1 = min(nb, d0 + per);
        int c = 0;
        for (int d = d0; d < d1; ++d) c += (int)hist[d];
        int tot;
        const int pre = block_exclusive_scan(c, s_scan, &tot);
        if (pre < need && pre + c >= need) {
            int acc = pre;
            for (int d = d0; d < d1; ++d) {
                if (acc + (int)hist[d] >= need) {
                    s_prefix = prefix | ((unsigned)d << sh);
                    s_need = need - acc;
                    s_at_thr = (int)hist[d];
                    break;
                }
                acc += (int)hist[d];
            }
        }
        __syncthreads();
        if (s_need == s_at_thr) {   // every key of the digit is taken
            lowmask = (1u << sh) - 1u;
            break;
        }
        if (lev == 0 && s_at_thr <= kSlCand) {
            cand = true;
            break;
        }
    }
    // selection.  Candidate path: keys of a first-level bin below the threshold's are taken, those of
    // its bin are ranked by (key, L index) and the first s_need taken.  Otherwise, when every key at
    // the threshold is taken (the usual case) one strided pass takes the keys up to it; else each
    // thread takes a contiguous run of groups of four L indices, ranked by a block scan.
    const unsigned thr = s_prefix | lowmask;
    const bool all = k >= ntot;
    const int take_eq = s_need;
    const bool whole = !cand && (all || take_eq == s_at_thr);
    if (cand) {
        const unsigned b0 = thr >> 20;
        for_each_key(sk4, nl4, tid, [&](unsigned key, int li) {
            if (key == ~0u) return;
            if ((key >> 20) < b0) {
                const int at = atomicAdd(&s_count, 1);
                if (at < kMaxShortlist) s_sel[at] = li;
            } else if ((key >> 20) == b0) {
                const int c = atomicAdd(&s_ncand, 1);
                if (c < kSlCand) s_cand[c] = make_uint2(key, (unsigned)li);
            }
        });
        __syncthreads();
        const int nc = min(s_ncand, kSlCand);
        for (int c = tid; c < nc; c += kSlThreads) {
            const uint2 me = s_cand[c];
            int r = 0;
            for (int o = 0; o < nc; ++o) {
                const uint2 ot = s_cand[o];
                r += (ot.x < me.x) || (ot.x == me.x && ot.y < me.y);
            }
            if (r < take_eq) {
                const int at = atomicAdd(&s_count, 1);
                if (at < kMaxShortlist) s_sel[at] = (int)me.y;
            }
        }
    }
    if (k > 0 && whole)
        for_each_key(sk4, nl4, tid, [&](unsigned key, int li) {
            if (key == ~0u || !(all || key <= thr)) return;
            const int at = atomicAdd(&s_count, 1);
            if (at < kMaxShortlist) s_sel[at] = li;
        });
    const int run = (nl4 + kSlThreads - 1) / kSlThreads;
    const int g0 = min(nl4, tid * run), g1 = min(nl4, g0 + run);
    int eq = 0;
    if (!whole && !cand && k > 0)
        for (int i4 = g0; i4 < g1; ++i4) {
            const uint4 kq = sk4[i4];
            eq += (kq.x == thr) + (kq.y == thr) + (kq.z == thr) + (kq.w == thr);
        }
    int eqtot;
    const int eqpre = block_exclusive_scan(eq, s_scan, &eqtot);
    if (k > 0 && !whole && !cand) {
        int e = eqpre;
        for (int i4 = g0; i4 < g1; ++i4) {
            const uint4 kq = sk4[i4];
            const unsigned kk[4] = {kq.x, kq.y, kq.z, kq.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const unsigned key = kk[u];
                if (key == ~0u) continue;
                bool sel = key < thr;
                if (key == thr) sel = e++ < take_eq;
                if (sel) {
                    const int at = atomicAdd(&s_count, 1);
                    if (at < kMaxShortlist) s_sel[at] = 4 * i4 + u;
                }
            }
        }
    }
    __syncthreads();
    const int cnt = min(s_count, kMaxShortlist);
    // exact logits of the shortlisted keys, read from the pinned host cache, four lanes per key
    const T* host = reinterpret_cast<const T*>(V.kv_host) + (int64_t)kv * n * 2 * kHeadDim;
    for (int j0 = 0; j0 < cnt; j0 += kSlThreads / 4) {
        const int j = j0 + tid / 4;
        const int li = j < cnt ? s_sel[j] : -1;
        const T* key = li >= 0 ? host + (int64_t)V.ltok[(int64_t)kv * n + li] * 2 * kHeadDim : nullptr;
        ff x[G];
        exact_logits_quad<T, G>(q + (int64_t)row0 * kHeadDim, key, tid & 3, a.inv_sqrt_d, x);
        if (key != nullptr && (tid & 3) == 0)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                tl[(int64_t)(row0 + g) * a.ws_n + li] = make_float2(x[g].hi, x[g].lo);
                atomicMax(&rows[row0 + g].m_tag, tag_max((unsigned)a.gen, x[g].hi));
            }
    }
    for (int j = tid; j < cnt; j += kSlThreads) slist[(int64_t)unit * kMaxShortlist + j] = s_sel[j];
    if (tid == 0) scount[unit] = cnt;
}

// Exact sketch: the L logits from the keys themselves.
template <typename T, int G>
__global__ void __launch_bounds__(kTile) score_exact_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                            RowState* __restrict__ rows, float2* __restrict__ tl,
                                                            float2* __restrict__ th, int n_ltiles)
{
    pdl_trigger();   // the decision kernel may start its independent prologue
    if (threadIdx.x == 0) tline_stamp(a.tline, 0, true);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.hrows[blockIdx.y] = 0;   // host rows of this call (attention)
        a.pf_cnt[blockIdx.y] = 0;   // rows the prefetch claims, and of them the attention reads
        a.pf_used[blockIdx.y] = 0;
        if (blockIdx.y == 0) *a.dprog = (unsigned long long)(unsigned)a.gen << 32;   // no row decided yet
    }
    if ((int)blockIdx.x >= n_ltiles) {
        score_h_tile<T, G>(views, q, a, rows, th, blockIdx.x - n_ltiles);
        return;
    }
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
        const float m = warp_max(mloc[g]);
        if ((threadIdx.x & 31) == 0 && m > -INFINITY)
            atomicMax(&rows[row_of(b, kv * G + g, a.Hq)].m_tag, tag_max((unsigned)a.gen, m));
    }
    (void)red;
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
    const float m = untag_max(R.m_tag, (unsigned)a.gen);
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
// Then lambda, a_i, v_i, b_i, eq. (7) and the no-fetch test (Algorithm 2, its certificate and no-fetch steps).
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
    // w = 0 (an underflowed weight) gives lambda = 1 and a = v = b = 0 exactly; returning early also
    // keeps zero numerators away from the division's slow path
    if (!(w > 0.f)) return {0.f, 0.f, 0.f};
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
        R.beta_f = bf;
        R.n_shrunk = 0;
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
        if (V.flags[(int64_t)kv * V.n + tok] == 0) {
            ++nf;
            atomicOr(&a.ebits[(int64_t)row * (a.ws_n / 32 + 1) + (tok >> 5)], 1u << (tok & 31));
        }
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
    {
        const GainParams gp = gain_params(R, a.ldelta);
        for (int j = threadIdx.x; j < P; j += blockDim.x) {
            if (j < nl) key[j] = gain_key(gain_num(coef_of(w[j], rr[j], bf), j, R.b_arg, gp), j);
            else key[j] = ~0ull;
        }
    }
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
// Fused decision for rows whose L fits on chip (|L| <= 8 x kDecideCap): one thread-block cluster
// of C CTAs per query row.  CTA c keeps the L entries [c S, (c + 1) S) of the row (S = ceil(|L|/C))
// in shared memory for every pass.  Sums are float-float per thread (or exact fixed point),
// block-reduced, and combined in rank order across the cluster through distributed shared memory,
// so all CTAs of a row take identical decisions.  Scalar double-precision work is done by one
// thread per CTA and broadcast (FP64 throughput is low on this part).
//   phase 0: w^ = exp(t^ - m) (also written to wl for the attention), r, gamma = w^(1-r)/r and
//            rho = r/(1-r); D, sum w^, sum w^(1-r), sum rho.
//   phase 1: Definition 2's fixed point by safeguarded Newton on G(beta) = beta (1 + R) - A - W,
//            started above the root (four times the all-interior solution).
//   phase 2: a_i, v_i, b_i; eq. (7); the no-fetch test (Algorithm 2, its certificate and no-fetch steps).
//   phase 3: gain keys (eq. (9)) and k* (eq. (10)) by a search over the 48-bit keys (gain
//            descending, L index ascending): per level, the remaining key range is split into at most
//            2048 bins of a power-of-two width (the first level spans the cluster's own key range); a
//            cluster-wide histogram
//            of counts, exact fixed-point sums of a_i and v_i and the max of b_i (plain 32-bit shared
//            atomics) gives the residual certificate at every bin boundary, so the bin holding the
//            k*-th key is found without sorting.  A bin of one key ends the search; a bin of at most
//            64 keys is finished by one warp (the keys gathered, sorted and scanned exactly).
//   phase 4: E = L_g[:k*] = the keys up to the k*-th, written as marks and a token list.
// --------------------------------------------------------------------------------------------
constexpr int kDecideThreads = 1024;
constexpr int kDecideStreamThreads = 512;   // streaming variant: two CTAs per multiprocessor
constexpr int kDecideCap = 8192;   // L entries per CTA
constexpr int kDecideMaxCluster = 16;  // 16 is a non-portable cluster size: used when the GPU can run it
constexpr int kDecideStreamMaxCluster = 8;
// k* search: keys of 31 gain bits and 18 index bits; each level splits the remaining key range into
// 2^11 bins
constexpr int kKeyBits = 49;
constexpr int kDecideMaxL = 1 << (kKeyBits - 31);   // the longest L a row may have on the fused decision
constexpr int kSearchBits = 11;
constexpr int kSearchLevels = 5;
constexpr int kSearchBins = 1 << kSearchBits;
// histogram fields per bin: count, max b, three 14-bit pieces of sum a, three of sum v
constexpr int kSearchFields = 8;
constexpr size_t kDecideHistSmem = (size_t)kSearchFields * kSearchBins * 4;
constexpr size_t kDecideSmem = (size_t)kDecideCap * 16 + kDecideHistSmem;
static_assert(kDecideCap * kDecideMaxCluster <= (1 << (kKeyBits - 31)), "L index must fit the key's low bits");

struct DecideSlot {
    ff v[8];
    float f[4];
    int i[4];
};

// The two largest b_i of a set and the (lowest) L index of the largest.
struct Top2 {
    float b1, b2;
    int arg;
};

__device__ __forceinline__ Top2 top2_merge(const Top2& x, const Top2& y)
{
    if (y.b1 > x.b1 || (y.b1 == x.b1 && y.arg < x.arg)) return {y.b1, fmaxf(y.b2, x.b1), y.arg};
    return {x.b1, fmaxf(x.b2, y.b1), x.arg};
}

__device__ __forceinline__ Top2 shfl_xor_top2(const Top2& x, int o)
{
    return {__shfl_xor_sync(0xffffffffu, x.b1, o), __shfl_xor_sync(0xffffffffu, x.b2, o),
            __shfl_xor_sync(0xffffffffu, x.arg, o)};
}

// Sort key of an L entry: ~bits(D g_i) (gain descending; g_i >= 0 so the sign bit is dropped), then
// the L index ascending.
__device__ __forceinline__ unsigned long long search_key(unsigned key32, int j)
{
    return ((unsigned long long)(key32 & 0x7fffffffu) << (kKeyBits - 31)) | (unsigned)j;
}

struct SearchAcc {
    unsigned long long a, v;  // fixed-point sums
    unsigned b, c;            // max b (ordered bits), count
};

// A CTA's proposal for the level's boundary: the residual after its first acceptable bin.
struct SearchProp {
    unsigned long long a, v;
    unsigned b, c, in_bin;
    int cand;                 // the bin (0x7fffffff: none in this CTA's slice)
};

__device__ __forceinline__ SearchAcc search_add(const SearchAcc& x, const SearchAcc& y)
{
    return {x.a + y.a, x.v + y.v, max(x.b, y.b), x.c + y.c};
}

__device__ __forceinline__ SearchAcc shfl_down_acc(const SearchAcc& x, int o)
{
    return {__shfl_down_sync(0xffffffffu, x.a, o), __shfl_down_sync(0xffffffffu, x.v, o),
            __shfl_down_sync(0xffffffffu, x.b, o), __shfl_down_sync(0xffffffffu, x.c, o)};
}

// Block-wide exclusive suffix (the combination over threads with a higher index).
__device__ SearchAcc block_suffix_search(const SearchAcc& mine, SearchAcc* sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const SearchAcc zero = {0ull, 0ull, 0u, 0u};
    SearchAcc x = mine;
    for (int o = 1; o < 32; o <<= 1) {
        const SearchAcc y = shfl_down_acc(x, o);
        if (lane + o < 32) x = search_add(x, y);
    }
    if (lane == 0) sh[warp] = x;   // warp total
    SearchAcc r = shfl_down_acc(x, 1);
    if (lane == 31) r = zero;
    __syncthreads();
    if (warp == 0) {
        // exclusive suffix over the warp totals
        SearchAcc t = lane < nw ? sh[lane] : zero;
        for (int o = 1; o < 32; o <<= 1) {
            const SearchAcc y = shfl_down_acc(t, o);
            if (lane + o < 32) t = search_add(t, y);
        }
        SearchAcc e = shfl_down_acc(t, 1);
        if (lane == 31) e = zero;
        __syncwarp();
        if (lane < nw) sh[32 + lane] = e;
    }
    __syncthreads();
    return search_add(r, sh[32 + warp]);
}

// Block-wide sums of N fp32 partials, returned as float-float in warp 0: a compensated warp
// reduction (the rounding error of every addition is carried along), then float-float across the
// warps (two barriers).
template <int N>
__device__ __forceinline__ void block_sum_f_w0(const float (&v)[N], ff (&out)[N], ff* scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    float s[N], e[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        s[k] = v[k];
        e[k] = 0.f;
    }
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const float y = __shfl_xor_sync(0xffffffffu, s[k], o), ye = __shfl_xor_sync(0xffffffffu, e[k], o);
            const ff t = two_sum(s[k], y);
            s[k] = t.hi;
            e[k] = __fadd_rn(__fadd_rn(e[k], ye), t.lo);
        }
    __syncthreads();
    if (lane == 0)
#pragma unroll
        for (int k = 0; k < N; ++k) scratch[warp * N + k] = fast_two_sum(s[k], e[k]);
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) out[k] = lane < nw ? scratch[lane * N + k] : ff{0.f, 0.f};
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int k = 0; k < N; ++k) out[k] = ff_add(out[k], shfl_xor_ff(out[k], o));
    }
}

// Thread 0 of every CTA has written slot[parity].v[0..nv) (and, for TOP2, its top-2 of b); warp 0
// reads them, one rank per lane, and combines them with a butterfly of symmetric operations, so
// every CTA of the cluster obtains bit-identical totals.
template <bool TOP2, bool EXT = false>
__device__ __forceinline__ void cluster_combine(cg::cluster_group& cl, DecideSlot* slot, int parity, int nv, ff* out,
                                                Top2* top, float* ext = nullptr)
{
    cl.sync();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        ff x[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        Top2 t = {0.f, 0.f, 0x7fffffff};
        unsigned e[4] = {0x7f800000u, 0x7f800000u, 0u, 0u};
        if (lane < (int)cl.num_blocks()) {
            const DecideSlot* rs = cl.map_shared_rank(slot, lane) + parity;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k < nv) x[k] = rs->v[k];
            if (TOP2) t = Top2{rs->f[0], rs->f[1], rs->i[0]};
            if (EXT)
#pragma unroll
                for (int k = 0; k < 4; ++k) e[k] = __float_as_uint(rs->f[k]);
        }
        for (int o = 1; o < kDecideMaxCluster; o <<= 1) {
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = ff_add(x[k], shfl_xor_ff(x[k], o));
            if (TOP2) t = top2_merge(t, shfl_xor_top2(t, o));
        }
        if (EXT) {
            e[0] = __reduce_min_sync(0xffffffffu, e[0]);
            e[1] = __reduce_min_sync(0xffffffffu, e[1]);
            e[2] = __reduce_max_sync(0xffffffffu, e[2]);
            e[3] = __reduce_max_sync(0xffffffffu, e[3]);
        }
        if (lane == 0) {
            for (int k = 0; k < nv; ++k) out[k] = x[k];
            if (TOP2) *top = t;
            if (EXT)
#pragma unroll
                for (int k = 0; k < 4; ++k) ext[k] = __uint_as_float(e[k]);
        }
    }
    __syncthreads();
}

// Scalars of one row, computed by thread 0 of each CTA and broadcast through shared memory.
struct DecideScalars {
    ff theta, lo, hi, D;
    float th_up, th_dn;        // theta rounded up / down: alpha >= theta <=> alpha >= th_up, gamma > theta <=> gamma > th_dn
    int done;
    float bf;                  // beta in fp32
    GainParams gp;
    int arg, no_fetch;
    float Df, ldf, sa_scale, sv_scale;  // fixed-point scales: a_i * sa_scale, v_i * sv_scale (totals ~2^40)
    // radix search state
    unsigned long long klo, khi;        // the key range still searched
    int rem_cnt;                        // keys below the current prefix range (removed)
    unsigned long long rest_a, rest_v;  // keys above the current prefix range (kept), fixed point
    unsigned int rest_b, rest_c;        // max b over them (ordered float bits), their count
    int kstar, found, in_bin;
    unsigned long long kkey;            // the k*-th smallest key
    // binary shrinkage: entries whose gamma key is below bin_kb get lambda = r; alpha enters the
    // fixed-point sums as alpha * fs1 * fs2 (below 2^40)
    unsigned long long bin_kb;
    int n_shrunk;
    float fs1, fs2;
};

// Key of gamma >= 0 in the binary-shrinkage order: ~bits(gamma) without the sign bit (gamma descending).
__device__ __forceinline__ unsigned gamma_key32(float ga) { return ~__float_as_uint(ga) & 0x7fffffffu; }

// A key of the boundary bin with its exact fixed-point a, v and b (ordered bits).
struct SmallCand {
    unsigned long long key, a, v;
    unsigned b, pad;
};
constexpr int kSmallBin = 64;   // boundary bins this small are finished by one warp

// theta >= 0 is a normalised float-float (hi = RN(hi + lo)), so the smallest float >= theta is hi, or
// the next float up when lo > 0; the largest float <= theta is hi, or the next float down when lo < 0.
__device__ __forceinline__ void set_theta(DecideScalars& sc, ff th)
{
    sc.theta = th;
    sc.th_up = th.lo > 0.f ? __uint_as_float(__float_as_uint(th.hi) + 1u) : th.hi;
    sc.th_dn = th.lo < 0.f ? __uint_as_float(__float_as_uint(th.hi) - 1u) : th.hi;
}

__device__ __forceinline__ unsigned int fmax_bits(float x) { return __float_as_uint(fmaxf(x, 0.f)); }

// A non-negative fp32 value below 2^42, rounded to an integer and split into three 14-bit pieces with
// fp32 arithmetic only (each step is exact: the value carries 24 significant bits).
__device__ __forceinline__ void fixed_pieces(float x, unsigned* p)
{
    const float h2 = floorf(x * 0x1p-28f);
    const float r2 = __fsub_rn(x, h2 * 0x1p28f);
    const float h1 = floorf(r2 * 0x1p-14f);
    const float r1 = rintf(__fsub_rn(r2, h1 * 0x1p14f));
    // rounding can carry r1 to 2^14; fold the carry so every piece stays below 2^14
    const float c1 = r1 >= 0x1p14f ? 1.f : 0.f;
    const float h1c = h1 + c1, r1c = r1 - c1 * 0x1p14f;
    const float c2 = h1c >= 0x1p14f ? 1.f : 0.f;
    p[0] = (unsigned)r1c;
    p[1] = (unsigned)(h1c - c2 * 0x1p14f);
    p[2] = (unsigned)(h2 + c2);
}

// Finish of the k* search when the boundary bin holds at most kSmallBin keys (run by warp 0 of every
// CTA of the cluster, which all obtain the same answer): the keys of the bin are copied from every
// CTA's list into `loc`, each is placed by its rank (the keys are distinct), and the residual after
// each is the level's outside rest plus the exact suffix sums of the keys after it; k* ends at the
// first boundary whose certificate is below eps.
__device__ __forceinline__ void finish_small(cg::cluster_group& cl, const SmallCand* cand, const int* ncand,
                                             SmallCand* loc, DecideScalars& sc, int C, float ldf, float Df,
                                             float inv_fa, float inv_fv, float eps_f)
{
    const int lane = threadIdx.x & 31;
    // offsets of each CTA's list
    const int cnt = lane < C ? *cl.map_shared_rank(ncand, lane) : 0;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int ntot = __shfl_sync(0xffffffffu, incl, 31);
    SmallCand mine[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = lane + 32 * h;
        int rk = 0, off = 0;
        for (int r = 0; r < C; ++r) {
            const int ex = __shfl_sync(0xffffffffu, incl - cnt, r);   // exclusive offset of rank r
            if (e >= ex) { rk = r; off = ex; }
        }
        mine[h] = SmallCand{~0ull, 0ull, 0ull, 0u, 0u};
        if (e < ntot) mine[h] = cl.map_shared_rank(cand, rk)[e - off];
    }
    // rank of each key among the candidates (keys are distinct), then the sorted copy in `loc`
    __shared__ unsigned long long keys_[kSmallBin];
    keys_[lane] = mine[0].key;
    keys_[lane + 32] = mine[1].key;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (lane + 32 * h >= ntot) continue;
        int rnk = 0;
        for (int q = 0; q < ntot; ++q) rnk += keys_[q] < mine[h].key;
        loc[rnk] = mine[h];
    }
    __syncwarp();
    unsigned long long av[2], vv[2];
    unsigned bb[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        av[h] = i < ntot ? loc[i].a : 0ull;
        vv[h] = i < ntot ? loc[i].v : 0ull;
        bb[h] = i < ntot ? loc[i].b : 0u;
    }
    // exclusive suffix (over larger keys) of a, v and max b
    unsigned long long sa[2], sv[2];
    unsigned sb_[2];
    {
        unsigned long long xa = av[1], xv = vv[1];
        unsigned xb = bb[1];
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long ya = __shfl_down_sync(0xffffffffu, xa, o), yv = __shfl_down_sync(0xffffffffu, xv, o);
            const unsigned yb = __shfl_down_sync(0xffffffffu, xb, o);
            if (lane + o < 32) { xa += ya; xv += yv; xb = max(xb, yb); }
        }
        const unsigned long long ta1 = __shfl_sync(0xffffffffu, xa, 0), tv1 = __shfl_sync(0xffffffffu, xv, 0);
        const unsigned tb1 = __shfl_sync(0xffffffffu, xb, 0);
        sa[1] = xa - av[1];
        sv[1] = xv - vv[1];
        sb_[1] = __shfl_down_sync(0xffffffffu, xb, 1);
        if (lane == 31) sb_[1] = 0u;
        unsigned long long za = av[0], zv = vv[0];
        unsigned zb = bb[0];
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long ya = __shfl_down_sync(0xffffffffu, za, o), yv = __shfl_down_sync(0xffffffffu, zv, o);
            const unsigned yb = __shfl_down_sync(0xffffffffu, zb, o);
            if (lane + o < 32) { za += ya; zv += yv; zb = max(zb, yb); }
        }
        unsigned nb0 = __shfl_down_sync(0xffffffffu, zb, 1);
        if (lane == 31) nb0 = 0u;
        sa[0] = za - av[0] + ta1;
        sv[0] = zv - vv[0] + tv1;
        sb_[0] = max(nb0, tb1);
    }
    // the first key whose residual (the keys after it, plus the rest above the bin) is accepted
    int best = 0x7fffffff;
#pragma unroll
    for (int h = 1; h >= 0; --h) {
        const int i = lane + 32 * h;
        if (i < ntot) {
            const unsigned long long A = sc.rest_a + sa[h], Vv = sc.rest_v + sv[h];
            const unsigned Bm = max(sc.rest_b, sb_[h]);
            const int after = (ntot - 1 - i) + (int)sc.rest_c;
            if (after > 0 && cert_f((float)A * inv_fa, (float)Vv * inv_fv, __uint_as_float(Bm), ldf, Df) < eps_f) best = i;
        }
    }
    best = __reduce_min_sync(0xffffffffu, best);
    if (best == 0x7fffffff) best = ntot - 1;   // the bin's last boundary was accepted at its level
    if (lane == 0) {
        sc.found = 1;
        sc.kstar = sc.rem_cnt + best + 1;
        sc.kkey = loc[best].key;
    }
}

// Finish of the binary-shrinkage search when the bin holding the end of the shrunk prefix has at most
// kSmallBin entries (warp 0 of every CTA, all with the same answer): the bin's entries, gathered from
// every CTA, are placed by rank (the keys are distinct); entry i passes when its gamma exceeds twice
// the bias before it (the prefix up to the bin, sc.rest_a, plus the exact fixed-point sum of alpha over
// the bin's entries before i).  The first entry of the bin passes by construction; the prefix ends at
// the first entry that fails, or with the bin.  SmallCand carries (key, fixed-point alpha, -, gamma bits).
__device__ __forceinline__ void finish_binary(cg::cluster_group& cl, const SmallCand* cand, const int* ncand,
                                              SmallCand* loc, DecideScalars& sc, int C, float fs1, float fs2)
{
    const int lane = threadIdx.x & 31;
    const int cnt = lane < C ? *cl.map_shared_rank(ncand, lane) : 0;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int ntot = __shfl_sync(0xffffffffu, incl, 31);
    SmallCand mine[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int e = lane + 32 * h;
        int rk = 0, off = 0;
        for (int r = 0; r < C; ++r) {
            const int ex = __shfl_sync(0xffffffffu, incl - cnt, r);
            if (e >= ex) { rk = r; off = ex; }
        }
        mine[h] = SmallCand{~0ull, 0ull, 0ull, 0u, 0u};
        if (e < ntot) mine[h] = cl.map_shared_rank(cand, rk)[e - off];
    }
    __shared__ unsigned long long bkeys_[kSmallBin];
    bkeys_[lane] = mine[0].key;
    bkeys_[lane + 32] = mine[1].key;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (lane + 32 * h >= ntot) continue;
        int rnk = 0;
        for (int q = 0; q < ntot; ++q) rnk += bkeys_[q] < mine[h].key;
        loc[rnk] = mine[h];
    }
    __syncwarp();
    unsigned long long av[2];
    float gv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        av[h] = i < ntot ? loc[i].a : 0ull;
        gv[h] = i < ntot ? __uint_as_float(loc[i].b) : 0.f;
    }
    // exclusive prefix of alpha over the bin's entries in key order
    unsigned long long x0 = av[0], x1 = av[1];
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (lane >= o) { x0 += y0; x1 += y1; }
    }
    const unsigned long long tot0 = __shfl_sync(0xffffffffu, x0, 31);
    const unsigned long long ex[2] = {sc.rest_a + x0 - av[0], sc.rest_a + tot0 + x1 - av[1]};
    int first_fail = 0x7fffffff;
#pragma unroll
    for (int h = 1; h >= 0; --h) {
        const int i = lane + 32 * h;
        if (i < ntot && !(__fmul_rn(__fmul_rn(gv[h], fs1), fs2) > 2.0f * (float)ex[h])) first_fail = i;
    }
    first_fail = __reduce_min_sync(0xffffffffu, first_fail);
    if (lane == 0) {
        const int p = first_fail == 0x7fffffff ? ntot : first_fail;
        sc.found = 1;
        sc.n_shrunk = sc.rem_cnt + p;
        sc.bin_kb = p < ntot ? loc[p].key : sc.khi;
    }
}

template <bool BINARY, bool STREAM>
__global__ void __launch_bounds__(STREAM ? kDecideStreamThreads : kDecideThreads, STREAM ? 2 : 1)
decide_kernel(Views views, DecodeArgs a,
                                                                   RowState* __restrict__ rows,
                                                                   const float2* __restrict__ tl,
                                                                   const float2* __restrict__ th,
                                                                   float* __restrict__ wl,
                                                                   int32_t* __restrict__ mark,
                                                                   int32_t* __restrict__ elist,
                                                                   unsigned long long* scratch)
{
    pdl_wait();      // the scoring kernel has completed (its logits, maxima and weight factors are visible)
    pdl_trigger();   // the next kernel (prefetch or attention) may start: the scoring kernel's results are complete
    if (threadIdx.x == 0) tline_stamp(a.tline, 1, true);
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int rank = (int)cl.block_rank();
    const int row = blockIdx.x / C;
    extern __shared__ __align__(16) unsigned char dsm[];
    // phases 0-1: w^, r, gamma, rho; phase 2 leaves b_i, r, a_i, v_i; phase 3: b_i, gain keys, scaled a_i,
    // scaled v_i; then the histogram
    float* sw = reinterpret_cast<float*>(dsm);
    float* sr = sw + kDecideCap;
    float* sg = sr + kDecideCap;
    float* sp = sg + kDecideCap;
    unsigned* skey = reinterpret_cast<unsigned*>(sr);
    float* sb = sw;
    float* sa_ = sg;
    float* sv_ = sp;
    // [kSearchFields][kSearchBins]; the streaming variant keeps no entries in shared memory
    unsigned* hist = STREAM ? reinterpret_cast<unsigned*>(dsm) : reinterpret_cast<unsigned*>(sp + kDecideCap);
    __shared__ DecideSlot slot[2];
    __shared__ ff bc[8];
    __shared__ ff redff[32 * 4];
    __shared__ Top2 stop2[32];
    __shared__ Top2 ctop;
    __shared__ unsigned sext[32][4];
    __shared__ SmallCand bcand[kSmallBin], bloc[kSmallBin];
    __shared__ int ncand;
    __shared__ float bext[4];
    __shared__ int redi[32];
    __shared__ DecideScalars sc;
    __shared__ int wcnt[2];
    __shared__ SearchAcc sacc[64];
    __shared__ SearchAcc ssum;   // this CTA's slice total at the current search level
    __shared__ SearchProp sprop;
    const int tid = threadIdx.x, T = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = T >> 5;
    constexpr int BPT = STREAM ? 4 : 2;   // histogram bins per thread when a CTA reads its slice of bins
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    const SlotView& V = views.v[b];
    RowState& R = rows[row];
    const int nl = V.counts[kv * 4 + 1], nh = V.counts[kv * 4 + 0] + V.n_tail;
    const int S = (nl + C - 1) / C;
    const int j0 = min(nl, rank * S), j1 = min(nl, j0 + S), ns = j1 - j0;
    const float* rl = V.rl + (int64_t)kv * V.n;
    // The streaming variant keeps an entry's state in global memory (L2) instead of shared memory and
    // reads it back in every pass, four entries per thread in flight.  Through phase 2 that state is w^
    // (the row of wl) and the KV head's r and ratios ((1 - r) / r, r / (1 - r)), shared by the query
    // rows of the head, from which alpha = w (1 - r), gamma = w (1 - r) / r and rho = r / (1 - r) are
    // formed with the operations phase 0 of the on-chip variant uses.  For the k* search (rows that
    // fetch) the key pass writes each entry's search state into two scratch rows -- the row's logits
    // in tl (dead once phase 0 has read them; float2 per entry) and the row of the full-row key buffer
    // (idle on this path; two float planes of ws_npow2 entries): tl = the fixed-point-scaled
    // (a_i, v_i), plane A = gain key, plane B = bits of b_i.  An entry is written and read back only by
    // the thread that owns it (entry i on thread i mod T, in every pass), so program order makes the
    // values visible.
    float* const wl_row = wl + (int64_t)row * a.ws_n + j0;
    const float* const rl_row = rl + j0;
    const float2* const lq_row = V.lq + (int64_t)kv * V.n + j0;
    float2* const st_row = const_cast<float2*>(tl) + (int64_t)row * a.ws_n + j0;
    float* const pa_row = reinterpret_cast<float*>(scratch + (int64_t)row * a.ws_npow2) + j0;
    float* const pb_row = reinterpret_cast<float*>(scratch + (int64_t)row * a.ws_npow2) + a.ws_npow2 + j0;
    constexpr int U = 4;
    // body(i, w^, alpha, gamma, rho) for every entry of the slice (rho only where NEED_RHO)
    auto pass = [&](auto&& body) {
        if (STREAM) {
            for (int g0 = 0; g0 < ns; g0 += U * T) {
                float wv[U], rv[U];
                float2 qv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    wv[u] = i < ns ? wl_row[i] : 0.f;
                    rv[u] = i < ns ? __ldg(rl_row + i) : 0.5f;
                    qv[u] = i < ns ? __ldg(lq_row + i) : make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    if (i < ns)
                        body(i, wv[u], __fmul_rn(wv[u], __fsub_rn(1.0f, rv[u])), __fmul_rn(wv[u], qv[u].x), qv[u].y);
                }
            }
        } else {
            for (int i = tid; i < ns; i += T) body(i, sw[i], sr[i], sg[i], sp[i]);
        }
    };
    int parity = 0;
    const bool timer = rank == 0 && tid == 0;
    unsigned long long t_prev = timer ? global_ns() : 0ull;
    auto stamp = [&](int k) {
        if (timer) {
            const unsigned long long t = global_ns();
            R.phase_ns[k] = (unsigned)(t - t_prev);
            t_prev = t;
        }
    };

    float m;   // the row maximum of the logits
    float acc_lo[4] = {0.f, 0.f, 0.f, 0.f};   // streaming variant: low parts of the phase-0 partials
    // ---- phase 0: weights and the row totals; this row's exact-set bitmap (left by the previous
    // call for its attention) is cleared for phase 4
    {
        {
            const int64_t stride = a.ws_n / 32 + 1;
            uint32_t* eb = a.ebits + (int64_t)row * stride;
            const int per = (int)((stride + C - 1) / C);
            for (int wi = rank * per + tid; wi < min((int)stride, (rank + 1) * per); wi += T) eb[wi] = 0u;
        }
        // per-thread partial sums in fp32, combined across the block and the cluster in float-float:
        // sum_L w^, sum_H w, sum alpha, sum rho
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float2* tlr = tl + (int64_t)row * a.ws_n + j0;
        const float* rlr = rl + j0;
        const float2* lqr = V.lq + (int64_t)kv * V.n + j0;
        float* wlr = wl + (int64_t)row * a.ws_n + j0;
        if (STREAM) {
            // any number of entries per thread: float-float partials (a thread may hold hundreds)
            m = untag_max(R.m_tag, (unsigned)a.gen);
            ff pw = {0.f, 0.f}, pa = {0.f, 0.f}, pr = {0.f, 0.f};
            for (int g0 = 0; g0 < ns; g0 += U * T) {
                float2 tv[U], qv[U];
                float rv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    tv[u] = i < ns ? __ldcg(tlr + i) : make_float2(0.f, 0.f);
                    rv[u] = i < ns ? __ldg(rlr + i) : 0.5f;
                    qv[u] = i < ns ? __ldg(lqr + i) : make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    if (i >= ns) break;
                    const float w = weight_of(tv[u], m);
                    const float al = __fmul_rn(w, __fsub_rn(1.0f, rv[u]));   // alpha = w (1 - r)
                    wlr[i] = w;
                    pw = ff_add_f(pw, w);
                    pa = ff_add_f(pa, al);
                    pr = ff_add_f(pr, qv[u].y);
                }
            }
            acc[0] = pw.hi;
            acc[2] = pa.hi;
            acc[3] = pr.hi;
            // the low parts join the compensated block sum as a second set of terms below
            acc_lo[0] = pw.lo;
            acc_lo[2] = pa.lo;
            acc_lo[3] = pr.lo;
        } else {
        // all loads of a thread issued before any is used
        float2 tv[8], qv[8];
        float rv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * T;
            rv[k] = i < ns ? rlr[i] : 0.f;
            qv[k] = i < ns ? lqr[i] : make_float2(0.f, 0.f);
            // the scoring kernel's output (it may have been running when this grid started): through L2
            tv[k] = i < ns ? __ldcg(tlr + i) : make_float2(0.f, 0.f);
        }
        m = untag_max(R.m_tag, (unsigned)a.gen);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * T;
            if (i >= ns) break;
            const float w = weight_of(tv[k], m);
            const float r = rv[k];
            const float al = __fmul_rn(w, __fsub_rn(1.0f, r));
            sw[i] = w;
            sr[i] = al;                      // alpha = w (1 - r)
            wlr[i] = w;
            sg[i] = __fmul_rn(w, qv[k].x);   // gamma = w (1 - r) / r
            sp[i] = qv[k].y;                 // rho = r / (1 - r)
            acc[0] = __fadd_rn(acc[0], w);
            acc[2] = __fadd_rn(acc[2], al);
            acc[3] = __fadd_rn(acc[3], qv[k].y);
        }
        }
        if (rank == 0) {
            const float2* thr = th + (int64_t)row * a.ws_n;
            for (int k0 = tid; k0 < nh; k0 += 4 * T) {
                float2 hv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) hv[u] = k0 + u * T < nh ? __ldcg(thr + k0 + u * T) : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (k0 + u * T < nh) acc[1] = __fadd_rn(acc[1], weight_of(hv[u], m));
            }
        }
        ff tot[4];
        block_sum_f_w0<4>(acc, tot, redff);
        if (STREAM) {
            ff tlo[4];
            block_sum_f_w0<4>(acc_lo, tlo, redff);
            if (warp == 0)
#pragma unroll
                for (int k = 0; k < 4; ++k) tot[k] = ff_add(tot[k], tlo[k]);
        }
        if (tid == 0) {
            for (int k = 0; k < 4; ++k) slot[parity].v[k] = tot[k];
            if (rank == 0) { wcnt[0] = 0; wcnt[1] = 0; }   // exact-list position and fetch count (phase 4)
        }
    }
    cluster_combine<false>(cl, slot, parity, 4, bc, nullptr);
    parity ^= 1;
    if (tid == 0) {
        const ff At = bc[2];
        const ff Dt = ff_add(bc[0], bc[1]);
        if (rank == 0) {
            R.D = ff_to_f64(Dt);
            R.alpha_sum = ff_to_f64(At);
            R.n_l = nl;
            R.n_h = nh;
            R.sel_passes = 0;
            for (int k = 0; k < 6; ++k) R.phase_ns[k] = 0;
        }
        sc.D = Dt;
        sc.lo = ff{0.f, 0.f};
        sc.hi = At;
        set_theta(sc, ff_min(At, ff_div(ff_mul_f(bc[0], 4.0f), ff_add_f(bc[3], 1.0f))));
        sc.done = (nl == 0 || !(At.hi > 0.f));
    }
    __syncthreads();
    stamp(0);

    int iters = 0;
    if (BINARY) {
        // ---- phase 1, binary shrinkage (Appendix A.2): in the order of decreasing gamma = w^ (1 - r) / r
        // (ties: lower L index), each entry gets lambda = r while its gamma exceeds twice the bias (sum
        // of alpha = w^ (1 - r)) of the entries before it.  Along the order gamma falls and the bias
        // grows, so the passing entries form a prefix.  Its end is searched like k* below, over the
        // gamma keys: per level a cluster-wide histogram of counts, exact fixed-point sums of alpha and
        // the largest gamma of every bin gives the test of each bin's first entry from the bias before
        // the bin; the last bin whose first entry passes holds the end (entries of gamma 0 never pass
        // and stay out).
        unsigned kmin = 0xffffffffu, kmax = 0u;
        pass([&](int i, float, float, float ga, float) {
            if (!(ga > 0.f)) return;
            const unsigned k32 = gamma_key32(ga);
            kmin = min(kmin, k32);
            kmax = max(kmax, k32);
        });
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        if (lane == 0) {
            sext[warp][0] = kmin;
            sext[warp][1] = kmax;
        }
        uint4* hist4 = reinterpret_cast<uint4*>(hist);
        for (int k = tid; k < kSearchFields * kSearchBins / 4; k += T) hist4[k] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        if (warp == 0) {
            kmin = __reduce_min_sync(0xffffffffu, lane < nw ? sext[lane][0] : 0xffffffffu);
            kmax = __reduce_max_sync(0xffffffffu, lane < nw ? sext[lane][1] : 0u);
            if (lane == 0) {
                slot[parity].i[0] = (int)kmin;
                slot[parity].i[1] = (int)kmax;
            }
        }
        cl.sync();   // every CTA's key range is published and every histogram is zero
        if (warp == 0) {
            const DecideSlot* rs = lane < C ? cl.map_shared_rank(slot, lane) + parity : nullptr;
            const unsigned mn = __reduce_min_sync(0xffffffffu, rs ? (unsigned)rs->i[0] : 0xffffffffu);
            const unsigned mx = __reduce_max_sync(0xffffffffu, rs ? (unsigned)rs->i[1] : 0u);
            if (lane == 0) {
                sc.done = 1;
                sc.rest_a = 0ull;
                sc.rem_cnt = 0;
                sc.in_bin = 0;
                sc.n_shrunk = 0;
                sc.bin_kb = 0ull;
                sc.fs1 = sc.fs2 = 1.0f;
                if (mn <= mx) {
                    sc.found = 0;
                    sc.klo = (unsigned long long)mn << (kKeyBits - 31);
                    sc.khi = ((unsigned long long)mx + 1ull) << (kKeyBits - 31);
                    // the largest gamma is below 2^E; alpha <= gamma is scaled by 2^(40 - E), split in two
                    // powers of two that are normal floats
                    const int E = (int)((0x7fffffffu - mn) >> 23) - 126;
                    const int k = 40 - E, k1 = k / 2, k2 = k - k1;
                    sc.fs1 = __int_as_float((127 + k1) << 23);
                    sc.fs2 = __int_as_float((127 + k2) << 23);
                } else {
                    sc.found = 1;   // no entry of positive gamma: nothing is shrunk
                }
            }
        }
        __syncthreads();
        parity ^= 1;
        const float fs1 = sc.fs1, fs2 = sc.fs2;
        const SearchAcc zero = {0ull, 0ull, 0u, 0u};
        for (int lev = 0; lev < kSearchLevels && !sc.found; ++lev) {
            ++iters;
            const int nb = kSearchBins;
            const int sl = nb / C;
            const unsigned long long klo = sc.klo, span = sc.khi - sc.klo;
            const int bs = max(0, (64 - __clzll((long long)(span - 1ull))) - kSearchBits);
            pass([&](int i, float, float al, float ga, float) {
                if (!(ga > 0.f)) return;
                const unsigned long long K = search_key(gamma_key32(ga), j0 + i);
                if (K < klo || K - klo >= span) return;
                const unsigned d = (unsigned)((K - klo) >> bs);
                unsigned pa[3];
                fixed_pieces(__fmul_rn(__fmul_rn(al, fs1), fs2), pa);
                atomicAdd(&hist[d], 1u);
                atomicMax(&hist[kSearchBins + d], __float_as_uint(ga));
#pragma unroll
                for (int q = 0; q < 3; ++q) atomicAdd(&hist[(2 + q) * kSearchBins + d], pa[q]);
            });
            __syncthreads();
            if (C > 1) {
                for (int d = tid; d < nb; d += T) {
                    const int ow = d / sl;
                    const unsigned cnt = hist[d];
                    if (ow == rank || cnt == 0u) continue;
                    unsigned* dst = cl.map_shared_rank(hist, ow);
                    atomicAdd(dst + d, cnt);
                    atomicMax(dst + kSearchBins + d, hist[kSearchBins + d]);
#pragma unroll
                    for (int f = 2; f < 5; ++f) atomicAdd(dst + f * kSearchBins + d, hist[f * kSearchBins + d]);
                }
                cl.sync();
            }
            // the cluster totals of this CTA's slice, BPT bins per thread in reverse order (thread t
            // holds bins dA = rank sl + sl - BPT (t + 1) .. dA + BPT - 1), so the threads above t hold
            // the bins before dA and the block's exclusive suffix is the prefix over bins
            const int dA = rank * sl + sl - BPT * (tid + 1);
            const bool own = BPT * (tid + 1) <= sl;
            unsigned c2[BPT], g2[BPT];
            unsigned long long a2[BPT];
            SearchAcc mine = zero;
#pragma unroll
            for (int k = 0; k < BPT; ++k) {
                c2[k] = g2[k] = 0u;
                a2[k] = 0ull;
                if (own) {
                    const int d = dA + k;
                    c2[k] = hist[d];
                    g2[k] = hist[kSearchBins + d];
#pragma unroll
                    for (int q = 0; q < 3; ++q) a2[k] += (unsigned long long)hist[(2 + q) * kSearchBins + d] << (14 * q);
                }
                mine.a += a2[k];
                mine.c += c2[k];
            }
            SearchAcc before = block_suffix_search(mine, sacc);
            if (tid == 0) ssum = search_add(before, mine);
            for (int k = tid; k < kSearchFields * kSearchBins / 4; k += T) hist4[k] = make_uint4(0u, 0u, 0u, 0u);
            cl.sync();
            // the slices before this one
            if (warp == 0) {
                SearchAcc x = (lane < rank) ? *cl.map_shared_rank(&ssum, lane) : zero;
                for (int o = 16; o > 0; o >>= 1) {
                    const SearchAcc y = {__shfl_xor_sync(0xffffffffu, x.a, o), __shfl_xor_sync(0xffffffffu, x.v, o),
                                         __shfl_xor_sync(0xffffffffu, x.b, o), __shfl_xor_sync(0xffffffffu, x.c, o)};
                    x = search_add(x, y);
                }
                if (lane == 0) sacc[0] = x;
            }
            __syncthreads();
            before = search_add(before, sacc[0]);
            // bias and count before the first entry of each of the thread's bins; the last bin whose
            // first entry passes
            unsigned long long Sk[BPT];
            unsigned nk[BPT];
            int mycand = -1;
#pragma unroll
            for (int k = 0; k < BPT; ++k) {
                Sk[k] = k == 0 ? sc.rest_a + before.a : Sk[k - 1] + a2[k - 1];
                nk[k] = k == 0 ? (unsigned)sc.rem_cnt + before.c : nk[k - 1] + c2[k - 1];
                const bool pk = c2[k] > 0u &&
                                __fmul_rn(__fmul_rn(__uint_as_float(g2[k]), fs1), fs2) > 2.0f * (float)Sk[k];
                if (own && pk) mycand = dA + k;
            }
            int cand = __reduce_max_sync(0xffffffffu, mycand);
            if (lane == 0) redi[warp] = cand;
            __syncthreads();
            cand = __reduce_max_sync(0xffffffffu, lane < nw ? redi[lane] : -1);
            if (own && cand >= dA && cand < dA + BPT) {
#pragma unroll
                for (int k = 0; k < BPT; ++k)
                    if (cand == dA + k) {
                        sprop.a = Sk[k];
                        sprop.c = nk[k];
                        sprop.in_bin = c2[k];
                    }
            }
            if (tid == 0) sprop.cand = cand;
            cl.sync();
            // the last bin of the level (highest CTA with a candidate) whose first entry passes
            if (warp == 0) {
                const int cr = lane < C ? cl.map_shared_rank(&sprop, lane)->cand : -1;
                const unsigned who = __ballot_sync(0xffffffffu, cr >= 0);
                if (lane == 0) {
                    if (who == 0u) {
                        // the range's first entry fails (only at the top level): nothing is shrunk
                        sc.found = 1;
                        sc.n_shrunk = sc.rem_cnt;
                        sc.bin_kb = klo;
                    } else {
                        const SearchProp p = *cl.map_shared_rank(&sprop, 31 - __clz(who));
                        sc.rest_a = p.a;
                        sc.rem_cnt = (int)p.c;
                        const unsigned long long d_ = (unsigned long long)p.cand;
                        sc.klo = klo + (d_ << bs);
                        sc.khi = min(klo + span, klo + ((d_ + 1ull) << bs));
                        sc.in_bin = (int)p.in_bin;
                        if (p.in_bin == 1u || lev == kSearchLevels - 1) {
                            sc.found = 1;
                            sc.n_shrunk = (int)(p.c + p.in_bin);
                            sc.bin_kb = sc.khi;
                        }
                    }
                }
            }
            __syncthreads();
            if (sc.found) break;
            if (sc.in_bin <= kSmallBin) {
                if (tid == 0) ncand = 0;
                __syncthreads();
                pass([&](int i, float, float al, float ga, float) {
                    if (!(ga > 0.f)) return;
                    const unsigned long long K = search_key(gamma_key32(ga), j0 + i);
                    if (K < sc.klo || K >= sc.khi) return;
                    const int at = atomicAdd(&ncand, 1);
                    unsigned pa[3];
                    fixed_pieces(__fmul_rn(__fmul_rn(al, fs1), fs2), pa);
                    bcand[at].key = K;
                    bcand[at].a = (unsigned long long)pa[0] + ((unsigned long long)pa[1] << 14) +
                                  ((unsigned long long)pa[2] << 28);
                    bcand[at].v = 0ull;
                    bcand[at].b = __float_as_uint(ga);
                });
                cl.sync();
                if (warp == 0) finish_binary(cl, bcand, &ncand, bloc, sc, C, fs1, fs2);
                __syncthreads();
                break;
            }
        }
    }

    // ---- phase 1: beta (Newton on the classes; thread 0 does the scalar update)
    while (!sc.done) {
        ++iters;
        const float tu = sc.th_up, td = sc.th_dn;
        float acc[3] = {0.f, 0.f, 0.f};  // A, W, R
        // the breakpoints nearest theta: min alpha of the lambda = r class, min gamma of the interior,
        // max alpha outside the lambda = r class, max gamma of the lambda = 1 class
        float uA = INFINITY, uG = INFINITY, lA = 0.f, lG = 0.f;
        ff accs[3] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};   // streaming variant: float-float partials
        pass([&](int i, float wj, float al, float ga, float rho) {
            if (!(wj > 0.f)) return;
            if (al >= tu) {                                   // theta <= alpha: lambda = r
                if (STREAM) accs[0] = ff_add_f(accs[0], al); else acc[0] = __fadd_rn(acc[0], al);
                uA = fminf(uA, al);
            } else {
                lA = fmaxf(lA, al);
                if (ga > td) {                                // theta < gamma: interior
                    if (STREAM) {
                        accs[1] = ff_add_f(accs[1], wj);
                        accs[2] = ff_add_f(accs[2], rho);
                    } else {
                        acc[1] = __fadd_rn(acc[1], wj);
                        acc[2] = __fadd_rn(acc[2], rho);
                    }
                    uG = fminf(uG, ga);
                } else {
                    lG = fmaxf(lG, ga);
                }
            }
        });
        {
            const unsigned e0 = __reduce_min_sync(0xffffffffu, __float_as_uint(uA));
            const unsigned e1 = __reduce_min_sync(0xffffffffu, __float_as_uint(uG));
            const unsigned e2 = __reduce_max_sync(0xffffffffu, __float_as_uint(lA));
            const unsigned e3 = __reduce_max_sync(0xffffffffu, __float_as_uint(lG));
            if (lane == 0) {
                sext[warp][0] = e0;
                sext[warp][1] = e1;
                sext[warp][2] = e2;
                sext[warp][3] = e3;
            }
        }
        ff tot[3];
        if (STREAM) {
            float hi3[3] = {accs[0].hi, accs[1].hi, accs[2].hi}, lo3[3] = {accs[0].lo, accs[1].lo, accs[2].lo};
            ff tlo[3];
            block_sum_f_w0<3>(hi3, tot, redff);   // its barriers also publish sext
            block_sum_f_w0<3>(lo3, tlo, redff);
            if (warp == 0)
#pragma unroll
                for (int k = 0; k < 3; ++k) tot[k] = ff_add(tot[k], tlo[k]);
        } else {
            block_sum_f_w0<3>(acc, tot, redff);   // its barriers also publish sext
        }
        if (warp == 0) {
            const unsigned e0 = __reduce_min_sync(0xffffffffu, lane < nw ? sext[lane][0] : 0x7f800000u);
            const unsigned e1 = __reduce_min_sync(0xffffffffu, lane < nw ? sext[lane][1] : 0x7f800000u);
            const unsigned e2 = __reduce_max_sync(0xffffffffu, lane < nw ? sext[lane][2] : 0u);
            const unsigned e3 = __reduce_max_sync(0xffffffffu, lane < nw ? sext[lane][3] : 0u);
            if (tid == 0) {
                for (int k = 0; k < 3; ++k) slot[parity].v[k] = tot[k];
                slot[parity].f[0] = __uint_as_float(e0);
                slot[parity].f[1] = __uint_as_float(e1);
                slot[parity].f[2] = __uint_as_float(e2);
                slot[parity].f[3] = __uint_as_float(e3);
            }
        }
        cluster_combine<false, true>(cl, slot, parity, 3, bc, nullptr, bext);
        parity ^= 1;
        if (tid == 0) {
            const ff theta = sc.theta;
            const ff AW = ff_add(bc[0], bc[1]), oneR = ff_add_f(bc[2], 1.0f);
            const ff g = ff_sub(ff_mul(theta, oneR), AW);
            if (g.hi >= 0.f) sc.hi = ff_min(sc.hi, theta); else sc.lo = ff_max(sc.lo, theta);
            ff nt = ff_div(AW, oneR);
            // the classes at nt are those at theta when no breakpoint lies between them: then nt is
            // the root (the next pass would return it again)
            const float nu_ = nt.lo > 0.f ? __uint_as_float(__float_as_uint(nt.hi) + 1u) : nt.hi;
            const float nd_ = nt.lo < 0.f ? __uint_as_float(__float_as_uint(nt.hi) - 1u) : nt.hi;
            const bool up = ff_lt(theta, nt);
            const bool same = up ? (bext[0] >= nu_ && bext[1] > nd_) : (bext[2] < nu_ && bext[3] <= nd_);
            if (same && !ff_eq(nt, theta) && ff_lt(sc.lo, nt) && ff_lt(nt, sc.hi)) {
                set_theta(sc, nt);
                sc.done = 1;
            } else if (ff_eq(nt, theta) || iters >= 200) sc.done = 1;
            else {
                if (!(ff_lt(sc.lo, nt) && ff_lt(nt, sc.hi)))
                    nt = sc.lo.hi > 0.f ? ff_sqrt(ff_mul(sc.lo, sc.hi)) : ff_mul_f(ff_add(sc.lo, sc.hi), 0.5f);
                if (ff_eq(nt, theta) || ff_sub(sc.hi, sc.lo).hi <= 0x1p-44f * sc.hi.hi) sc.done = 1;
                set_theta(sc, nt);
            }
        }
        __syncthreads();
    }
    if (tid == 0) {
        if (nl == 0) sc.theta = ff{0.f, 0.f};
        sc.bf = sc.theta.hi;
    }
    __syncthreads();
    const float bf = sc.bf;
    const unsigned long long bkb = BINARY ? sc.bin_kb : 0ull;
    stamp(1);
    // lambda, a_i, v_i, b_i of entry i and, for a sampled entry, its weight factor.  With alpha =
    // w (1 - r), gamma = alpha / r, rho = r / (1 - r):
    //   beta <= alpha: lambda = r, a = alpha, lambda w = w - alpha, v = lambda w alpha,
    //                  b = max(lambda w, alpha), weight factor 1;
    //   otherwise:     lambda = min(beta / gamma, 1), a = w - lambda w, v = lambda (lambda w) gamma,
    //                  b = max(lambda w, lambda gamma), weight factor lambda (1 + rho) / rho
    // (binary shrinkage: lambda = r on the passing prefix of the gamma order, 1 elsewhere)
    auto coef_entry = [&](int i, float w, float al, float gam, float rho, bool sampled, float& om_i) -> Coef {
        Coef c = {0.f, 0.f, 0.f};
        om_i = 1.0f;
        const bool at_r = BINARY ? (gam > 0.f && search_key(gamma_key32(gam), j0 + i) < bkb) : (bf <= al);
        if (!(w > 0.f)) {
            if (sampled) om_i = __fdiv_rn(__fadd_rn(1.0f, rho), rho);   // lambda = 1: 1 / r
        } else if (at_r) {
            const float lw = __fsub_rn(w, al);
            c.a = al;
            c.v = __fmul_rn(lw, al);
            c.b = fmaxf(lw, al);
        } else {
            const float lam = BINARY ? 1.0f : fminf(__fdiv_rn(bf, gam), 1.0f);
            const float lw = __fmul_rn(lam, w);
            c.a = __fsub_rn(w, lw);
            c.v = __fmul_rn(__fmul_rn(lam, lw), gam);
            c.b = fmaxf(lw, __fmul_rn(lam, gam));
            if (sampled) om_i = __fdiv_rn(__fmul_rn(lam, __fadd_rn(1.0f, rho)), rho);
        }
        return c;
    };

    // ---- phase 2: lambda, a_i, v_i, b_i and eq. (7); the weight factor lambda_i / r_i of the
    // sampled entries.  a, v, b replace gamma, rho, w^ in shared memory.
    {
        float acc[2] = {0.f, 0.f};
        Top2 t2 = {0.f, 0.f, 0x7fffffff};
        float* omr = a.om + (int64_t)row * a.ws_n;
        auto top2_add = [&](float bv, int j) {
            if (bv > t2.b1 || (bv == t2.b1 && j < t2.arg)) { t2.b2 = t2.b1; t2.b1 = bv; t2.arg = j; }
            else if (bv > t2.b2) t2.b2 = bv;
        };
        ff acc2[2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (STREAM) {
            const int32_t* ls_row = V.lslot + (int64_t)kv * V.n + j0;
            for (int g0 = 0; g0 < ns; g0 += U * T) {
                float wv[U], rv[U];
                float2 qv[U];
                int sv_[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    wv[u] = i < ns ? wl_row[i] : 0.f;
                    rv[u] = i < ns ? __ldg(rl_row + i) : 0.5f;
                    qv[u] = i < ns ? __ldg(lq_row + i) : make_float2(0.f, 0.f);
                    sv_[u] = i < ns ? __ldg(ls_row + i) : -1;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    if (i >= ns) break;
                    float om_i;
                    const Coef c = coef_entry(i, wv[u], __fmul_rn(wv[u], __fsub_rn(1.0f, rv[u])),
                                              __fmul_rn(wv[u], qv[u].x), qv[u].y, sv_[u] >= 0, om_i);
                    if (sv_[u] >= 0) omr[sv_[u]] = om_i;
                    acc2[0] = ff_add_f(acc2[0], c.a);
                    acc2[1] = ff_add_f(acc2[1], c.v);
                    top2_add(c.b, j0 + i);
                }
            }
            acc[0] = acc2[0].hi;
            acc[1] = acc2[1].hi;
        } else {
        int slv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * T;
            slv[k] = i < ns ? V.lslot[(int64_t)kv * V.n + j0 + i] : -1;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * T;
            if (i >= ns) break;
            float om_i;
            const Coef c = coef_entry(i, sw[i], sr[i], sg[i], sp[i], slv[k] >= 0, om_i);
            if (slv[k] >= 0) omr[slv[k]] = om_i;
            sg[i] = c.a;
            sp[i] = c.v;
            sw[i] = c.b;
            acc[0] = __fadd_rn(acc[0], c.a);
            acc[1] = __fadd_rn(acc[1], c.v);
            top2_add(c.b, j0 + i);
        }
        }
        for (int o = 16; o > 0; o >>= 1) t2 = top2_merge(t2, shfl_xor_top2(t2, o));
        if (lane == 0) stop2[warp] = t2;
        ff tot[2];
        block_sum_f_w0<2>(acc, tot, redff);   // its barriers also publish stop2
        if (STREAM) {
            float lo2[2] = {acc2[0].lo, acc2[1].lo};
            ff tlo[2];
            block_sum_f_w0<2>(lo2, tlo, redff);
            if (warp == 0) {
                tot[0] = ff_add(tot[0], tlo[0]);
                tot[1] = ff_add(tot[1], tlo[1]);
            }
        }
        if (warp == 0) {
            Top2 x = lane < nw ? stop2[lane] : Top2{0.f, 0.f, 0x7fffffff};
            for (int o = 16; o > 0; o >>= 1) x = top2_merge(x, shfl_xor_top2(x, o));
            if (tid == 0) {
                slot[parity].v[0] = tot[0];
                slot[parity].v[1] = tot[1];
                slot[parity].f[0] = x.b1;
                slot[parity].f[1] = x.b2;
                slot[parity].i[0] = x.arg;
            }
        }
    }
    cluster_combine<true>(cl, slot, parity, 2, bc, &ctop);
    if (tid == 0) {
        // the two largest b across the cluster (lowest index among equal maxima)
        const Top2 x = ctop;
        const float B1 = x.b1, B2 = nl > 1 ? x.b2 : 0.f;
        const ff SA = bc[0], SV = bc[1], ld = a.ld_ff;
        const ff three = {3.0f, 0.f};
        const ff t3 = ff_div(ff_mul_f(ld, B1), three);
        const ff Aq = ff_add(ff_mul(t3, t3), ff_mul_f(ff_mul(SV, ld), 2.0f));
        const ff sq = ff_sqrt(Aq);
        const ff eh = nl > 0 ? ff_div(ff_add(ff_add(SA, t3), sq), sc.D) : ff{0.f, 0.f};
        const bool nof = ff_lt(eh, a.eps_ff);
        sc.no_fetch = nof || nl == 0;
        sc.arg = x.arg;
        const ff t2 = ff_div(ff_mul_f(ld, B2), three);
        sc.gp.t = t3.hi;
        sc.gp.tm2 = t2.hi;
        sc.gp.A = Aq.hi;
        sc.gp.sqrtA = sq.hi;
        sc.gp.ld2 = __fmul_rn(2.0f, ld.hi);
        sc.ldf = ld.hi;
        sc.Df = sc.D.hi;
        sc.sa_scale = SA.hi > 0.f ? __fdiv_rn(0x1p40f, SA.hi) : 0.f;
        sc.sv_scale = SV.hi > 0.f ? __fdiv_rn(0x1p40f, SV.hi) : 0.f;
        sc.klo = 0;
        sc.khi = 0;
        sc.rem_cnt = 0;
        sc.rest_a = 0;
        sc.rest_v = 0;
        sc.rest_b = 0;
        sc.rest_c = 0;
        sc.found = 0;
        sc.kstar = nl;
        sc.kkey = ~0ull;
        if (rank == 0) {
            R.beta = BINARY ? ff_to_f64(SA) : ff_to_f64(sc.theta);   // binary: the bias of the coefficients
            R.beta_f = BINARY ? SA.hi : bf;
            R.n_shrunk = BINARY ? sc.n_shrunk : 0;
            R.sum_a = ff_to_f64(SA);
            R.V = ff_to_f64(SV);
            R.b1 = nl > 0 ? f32_to_f64_bits(B1) : 0.0;
            R.b2 = f32_to_f64_bits(B2);
            R.b_arg = nl > 0 ? x.arg : -1;
            R.eps_hat = ff_to_f64(eh);
            R.no_fetch = nof;
            R.kstar = 0;
            R.fallback = 0;
            R.n_fetch = 0;
            R.beta_iters = iters;
        }
    }
    parity ^= 1;
    __syncthreads();
    stamp(2);
    if (!sc.no_fetch) {
    const GainParams gp = sc.gp;
    const int ARG = sc.arg;
    const float fa = sc.sa_scale, fv = sc.sv_scale;
    // f(i, k32, sa, sv, bb) for every entry of the slice: its 32-bit gain key (~bits of D g_i), its
    // fixed-point-scaled a_i and v_i and the ordered bits of b_i (read from shared memory after the key
    // pass, recomputed from w^, r and beta by the streaming variant)
    auto search_pass = [&](auto&& f) {
        if (STREAM) {
            for (int g0 = 0; g0 < ns; g0 += U * T) {
                float2 av[U];
                unsigned kv_[U], bv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    av[u] = i < ns ? st_row[i] : make_float2(0.f, 0.f);
                    kv_[u] = i < ns ? __float_as_uint(pa_row[i]) : 0u;
                    bv[u] = i < ns ? __float_as_uint(pb_row[i]) : 0u;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    if (i < ns) f(i, kv_[u], av[u].x, av[u].y, bv[u]);
                }
            }
        } else {
            for (int i = tid; i < ns; i += T) f(i, skey[i], sa_[i], sv_[i], fmax_bits(sb[i]));
        }
    };

    // ---- phase 3: gain keys, then k* by the radix search
    {
        // entries of gain exactly 0 (an underflowed weight: a = v = 0) end every order and never move
        // k*: they stay out of the search, counted (with their max b) in every residual
        unsigned kmin = 0xffffffffu, kmax = 0u, zc = 0u, zb = 0u;
        auto range = [&](unsigned k32, unsigned bb) {
            if ((k32 & 0x7fffffffu) == 0x7fffffffu) {
                ++zc;
                zb = max(zb, bb);
            } else {
                kmin = min(kmin, k32 & 0x7fffffffu);
                kmax = max(kmax, k32 & 0x7fffffffu);
            }
        };
        if (STREAM) {
            // a_i, v_i, b_i recomputed from w^, r and beta (rows that fetch nothing never get here)
            pass([&](int i, float w, float al, float gam, float rho) {
                float om_;
                const Coef c = coef_entry(i, w, al, gam, rho, false, om_);
                const unsigned k32 = ~__float_as_uint(gain_num(c, j0 + i, ARG, gp));
                const unsigned bb = fmax_bits(c.b);
                st_row[i] = make_float2(__fmul_rn(c.a, fa), __fmul_rn(c.v, fv));
                pa_row[i] = __uint_as_float(k32);
                pb_row[i] = __uint_as_float(bb);
                range(k32, bb);
            });
        } else {
            for (int i = tid; i < ns; i += T) {
                Coef c;
                c.a = sg[i];
                c.v = sp[i];
                const unsigned k32 = ~__float_as_uint(gain_num(c, j0 + i, ARG, gp));
                skey[i] = k32;
                sa_[i] = __fmul_rn(c.a, fa);   // fixed-point-scaled a_i, v_i (exactly converted below)
                sv_[i] = __fmul_rn(c.v, fv);
                range(k32, fmax_bits(sb[i]));
            }
        }
        // the cluster's range of the other keys: the first search level spreads its bins over it
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        zc = __reduce_add_sync(0xffffffffu, zc);
        zb = __reduce_max_sync(0xffffffffu, zb);
        if (lane == 0) {
            sext[warp][0] = kmin;
            sext[warp][1] = kmax;
            sext[warp][2] = zc;
            sext[warp][3] = zb;
        }
        __syncthreads();
        if (warp == 0) {
            kmin = __reduce_min_sync(0xffffffffu, lane < nw ? sext[lane][0] : 0xffffffffu);
            kmax = __reduce_max_sync(0xffffffffu, lane < nw ? sext[lane][1] : 0u);
            zc = __reduce_add_sync(0xffffffffu, lane < nw ? sext[lane][2] : 0u);
            zb = __reduce_max_sync(0xffffffffu, lane < nw ? sext[lane][3] : 0u);
            if (lane == 0) {
                slot[parity].i[0] = (int)kmin;
                slot[parity].i[1] = (int)kmax;
                slot[parity].i[2] = (int)zc;
                slot[parity].i[3] = (int)zb;
            }
        }
    }
    stamp(3);
    {
        const float ldf = sc.ldf, Df = sc.Df, inv_fa = sc.sa_scale > 0.f ? 1.0f / sc.sa_scale : 0.f,
                    inv_fv = sc.sv_scale > 0.f ? 1.0f / sc.sv_scale : 0.f;
        const SearchAcc zero = {0ull, 0ull, 0u, 0u};
        int passes = 0;
        uint4* hist4 = reinterpret_cast<uint4*>(hist);
        for (int k = tid; k < kSearchFields * kSearchBins / 4; k += T) hist4[k] = make_uint4(0u, 0u, 0u, 0u);
        cl.sync();   // every histogram of the cluster is zero before any CTA adds to a remote one
        if (warp == 0) {
            const DecideSlot* rs = lane < C ? cl.map_shared_rank(slot, lane) + parity : nullptr;
            const unsigned mn = __reduce_min_sync(0xffffffffu, rs ? (unsigned)rs->i[0] : 0xffffffffu);
            const unsigned mx = __reduce_max_sync(0xffffffffu, rs ? (unsigned)rs->i[1] : 0u);
            const unsigned zc = __reduce_add_sync(0xffffffffu, rs ? (unsigned)rs->i[2] : 0u);
            const unsigned zb = __reduce_max_sync(0xffffffffu, rs ? (unsigned)rs->i[3] : 0u);
            if (lane == 0) {
                if (mn <= mx) {
                    sc.klo = (unsigned long long)mn << (kKeyBits - 31);
                    sc.khi = ((unsigned long long)mx + 1ull) << (kKeyBits - 31);
                } else {
                    sc.klo = sc.khi = 0ull;   // no key of positive gain: the search finds no boundary
                }
                sc.rest_c = zc;
                sc.rest_b = zb;
            }
        }
        __syncthreads();
        parity ^= 1;
        // each level splits the current key range [klo, khi) into bins of 2^bs keys (K falls in bin
        // (K - klo) >> bs, at most kSearchBins of them); a level shrinks the range by at least
        // kSearchBins / 2, so five levels reach a single key
        for (int lev = 0; lev < kSearchLevels; ++lev) {
            ++passes;
            const int nb = kSearchBins;
            const int sl = nb / C;   // bins per slice: CTA r owns the cluster totals of bins [r sl, (r + 1) sl)
            const unsigned long long klo = sc.klo, span = sc.khi - sc.klo;
            // bins of 2^bs keys, bs the smallest shift that fits the range in nb bins (at least half used)
            const int bs = max(0, (64 - __clzll((long long)(span - 1ull))) - kSearchBits);
            search_pass([&](int i, unsigned k32, float sa, float sv, unsigned bb) {
                const unsigned long long K = search_key(k32, j0 + i);
                if (K < klo || K - klo >= span) return;
                const unsigned d = (unsigned)((K - klo) >> bs);
                unsigned pa[3], pv[3];
                fixed_pieces(sa, pa);
                fixed_pieces(sv, pv);
                atomicAdd(&hist[d], 1u);
                atomicMax(&hist[kSearchBins + d], bb);
#pragma unroll
                for (int q = 0; q < 3; ++q) {
                    atomicAdd(&hist[(2 + q) * kSearchBins + d], pa[q]);
                    atomicAdd(&hist[(5 + q) * kSearchBins + d], pv[q]);
                }
            });
            __syncthreads();
            if (C > 1) {
                // add the non-empty bins of the other slices into their owners' histograms
                for (int d = tid; d < nb; d += T) {
                    const int ow = d / sl;
                    const unsigned cnt = hist[d];
                    if (ow == rank || cnt == 0u) continue;
                    unsigned* dst = cl.map_shared_rank(hist, ow);
                    atomicAdd(dst + d, cnt);
                    atomicMax(dst + kSearchBins + d, hist[kSearchBins + d]);
#pragma unroll
                    for (int f = 2; f < kSearchFields; ++f) atomicAdd(dst + f * kSearchBins + d, hist[f * kSearchBins + d]);
                }
                cl.sync();
            }
            // cluster totals of this CTA's bins d0 = rank sl + BPT tid .. d0 + BPT - 1
            const int d0 = rank * sl + BPT * tid;
            unsigned c2[BPT], b2[BPT];
            unsigned long long a2[BPT], v2[BPT];
            SearchAcc mine = zero;
#pragma unroll
            for (int k = 0; k < BPT; ++k) {
                c2[k] = b2[k] = 0u;
                a2[k] = v2[k] = 0ull;
                if (BPT * tid + k < sl) {
                    const int d = d0 + k;
                    c2[k] = hist[d];
                    b2[k] = hist[kSearchBins + d];
#pragma unroll
                    for (int q = 0; q < 3; ++q) {
                        a2[k] += (unsigned long long)hist[(2 + q) * kSearchBins + d] << (14 * q);
                        v2[k] += (unsigned long long)hist[(5 + q) * kSearchBins + d] << (14 * q);
                    }
                }
                mine = search_add(mine, SearchAcc{a2[k], v2[k], b2[k], c2[k]});
            }
            // exclusive suffix within the slice (higher bins = smaller gains); the slice total goes out
            SearchAcc above = block_suffix_search(mine, sacc);
            if (tid == 0) ssum = search_add(above, mine);
            // the histogram is consumed: clear it for the next level
            for (int k = tid; k < kSearchFields * kSearchBins / 4; k += T) hist4[k] = make_uint4(0u, 0u, 0u, 0u);
            cl.sync();
            // the slices above this one, then the keys above the level's range
            if (warp == 0) {
                SearchAcc x = (lane > rank && lane < C) ? *cl.map_shared_rank(&ssum, lane) : zero;
                for (int o = 16; o > 0; o >>= 1) {
                    const SearchAcc y = {__shfl_xor_sync(0xffffffffu, x.a, o), __shfl_xor_sync(0xffffffffu, x.v, o),
                                         __shfl_xor_sync(0xffffffffu, x.b, o), __shfl_xor_sync(0xffffffffu, x.c, o)};
                    x = search_add(x, y);
                }
                if (lane == 0) sacc[0] = x;
            }
            __syncthreads();
            above = search_add(above, sacc[0]);
            above.a += sc.rest_a;
            above.v += sc.rest_v;
            above.b = max(above.b, sc.rest_b);
            above.c += sc.rest_c;
            // residual after bin d0 + BPT - 1 = above; after bin d0 + k = after bin d0 + k + 1 plus that bin
            SearchAcc after[BPT];
            after[BPT - 1] = above;
#pragma unroll
            for (int k = BPT - 2; k >= 0; --k) after[k] = search_add(after[k + 1], SearchAcc{a2[k + 1], v2[k + 1], b2[k + 1], c2[k + 1]});
            int cand = 0x7fffffff;
#pragma unroll
            for (int k = BPT - 1; k >= 0; --k) {
                if (c2[k] > 0 && after[k].c > 0) {
                    const float A_ = (float)after[k].a * inv_fa, V_ = (float)after[k].v * inv_fv;
                    if (cert_f(A_, V_, __uint_as_float(after[k].b), ldf, Df) < a.eps_f) cand = d0 + k;
                }
            }
            cand = __reduce_min_sync(0xffffffffu, cand);
            if (lane == 0) redi[warp] = cand;
            __syncthreads();
            cand = __reduce_min_sync(0xffffffffu, lane < nw ? redi[lane] : 0x7fffffff);
            if (cand != 0x7fffffff && (cand - rank * sl) / BPT == tid) {
#pragma unroll
                for (int k = 0; k < BPT; ++k)
                    if (cand == d0 + k) {
                        sprop.a = after[k].a;
                        sprop.v = after[k].v;
                        sprop.b = after[k].b;
                        sprop.c = after[k].c;
                        sprop.in_bin = c2[k];
                    }
            }
            if (tid == 0) sprop.cand = cand;
            cl.sync();
            // the first bin of the level (lowest CTA with a candidate) whose residual is acceptable
            if (warp == 0) {
                const int cr = lane < C ? cl.map_shared_rank(&sprop, lane)->cand : 0x7fffffff;
                const unsigned who = __ballot_sync(0xffffffffu, cr != 0x7fffffff);
                if (lane == 0) {
                    if (who == 0u) {
                        // no boundary of the range leaves an acceptable non-empty residual: every key is
                        // taken (only possible at the top level: eps^(empty) = 0 is always accepted)
                        sc.found = 1;
                        sc.kstar = nl;
                        sc.kkey = ~0ull;
                    } else {
                        const SearchProp p = *cl.map_shared_rank(&sprop, __ffs(who) - 1);
                        sc.rest_a = p.a;
                        sc.rest_v = p.v;
                        sc.rest_b = p.b;
                        sc.rest_c = p.c;
                        sc.rem_cnt = nl - (int)p.in_bin - (int)p.c;
                        const unsigned long long d_ = (unsigned long long)p.cand;
                        sc.klo = klo + (d_ << bs);
                        sc.khi = min(klo + span, klo + ((d_ + 1ull) << bs));
                        sc.in_bin = (int)p.in_bin;
                        if (p.in_bin == 1u || lev == kSearchLevels - 1) {
                            // one key left (or, defensively, the whole bin at the last level)
                            sc.found = 1;
                            sc.kstar = sc.rem_cnt + (int)p.in_bin;
                            sc.kkey = sc.khi - 1ull;
                        }
                    }
                }
            }
            __syncthreads();
            if (sc.found) break;
            if (sc.in_bin <= kSmallBin) {
                // few keys left in the boundary bin: gather them, sort them and scan them directly
                if (tid == 0) ncand = 0;
                __syncthreads();
                search_pass([&](int i, unsigned k32, float sa, float sv, unsigned bb) {
                    const unsigned long long K = search_key(k32, j0 + i);
                    if (K < sc.klo || K >= sc.khi) return;
                    const int at = atomicAdd(&ncand, 1);
                    unsigned pa[3], pv[3];
                    fixed_pieces(sa, pa);
                    fixed_pieces(sv, pv);
                    bcand[at].key = K;
                    bcand[at].a = (unsigned long long)pa[0] + ((unsigned long long)pa[1] << 14) +
                                 ((unsigned long long)pa[2] << 28);
                    bcand[at].v = (unsigned long long)pv[0] + ((unsigned long long)pv[1] << 14) +
                                 ((unsigned long long)pv[2] << 28);
                    bcand[at].b = bb;
                });
                cl.sync();
                if (warp == 0) finish_small(cl, bcand, &ncand, bloc, sc, C, ldf, Df, inv_fa, inv_fv, a.eps_f);
                __syncthreads();
                break;
            }
        }
        if (timer) R.sel_passes = passes;
    }
    stamp(4);

    // ---- phase 4: E = keys up to the k*-th; each CTA writes its own members, claiming positions of
    // the exact list (whose order is irrelevant) and counting fetched tokens on rank 0's counters
    {
        const unsigned long long kk = sc.kkey;
        static_assert(kDecideCap == 8 * kDecideThreads, "emit assumes eight entries per thread");
        int* pos0 = cl.map_shared_rank(&wcnt[0], 0);
        int nf = 0;
        int32_t* el = elist + (int64_t)row * a.ws_n;
        uint32_t* eb = a.ebits + (int64_t)row * (a.ws_n / 32 + 1);
        float* omr = a.om + (int64_t)row * a.ws_n;
        // one selected entry: its list position (claimed per warp), weight factor 1 if sampled, else a
        // bit of the fetch bitmap
        auto emit = [&](bool sel, int tok, int slt) {
            const unsigned m8 = __ballot_sync(0xffffffffu, sel);
            if (m8 == 0u) return;
            int base = 0;
            if (lane == __ffs(m8) - 1) base = atomicAdd(pos0, __popc(m8));
            base = __shfl_sync(0xffffffffu, base, __ffs(m8) - 1);
            if (sel) {
                el[base + __popc(m8 & ((1u << lane) - 1u))] = tok;
                if (slt >= 0) {
                    omr[slt] = 1.0f;   // sampled and made exact: weight factor 1
                } else {
                    ++nf;
                    atomicOr(&eb[tok >> 5], 1u << (tok & 31));
                }
            }
        };
        if (STREAM) {
            // a warp-uniform trip count: the ballots of emit need every lane
            for (int g0 = 0; g0 < ns; g0 += U * T) {
                unsigned kv_[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    kv_[u] = i < ns ? __float_as_uint(pa_row[i]) : 0u;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = g0 + u * T + tid;
                    const bool sel = i < ns && search_key(kv_[u], j0 + i) <= kk;
                    const int64_t e = (int64_t)kv * V.n + j0 + i;
                    emit(sel, sel ? V.ltok[e] : 0, sel ? V.lslot[e] : -1);
                }
            }
        } else {
        bool sel[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = tid + k * T;
            sel[k] = i < ns && search_key(skey[i], j0 + i) <= kk;
        }
        // tokens and resident slots of the selected entries: all loads issued before any is used
        int tok[8], sl8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t e = (int64_t)kv * V.n + j0 + tid + k * T;
            tok[k] = sel[k] ? V.ltok[e] : 0;
            sl8[k] = sel[k] ? V.lslot[e] : -1;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) emit(sel[k], tok[k], sl8[k]);
        }
        nf = __reduce_add_sync(0xffffffffu, (unsigned)nf);
        if (lane == 0 && nf > 0) atomicAdd(cl.map_shared_rank(&wcnt[1], 0), nf);
        cl.sync();   // every CTA's additions to rank 0's counters are done (and no CTA leaves early)
        if (rank == 0 && tid == 0) {
            R.kstar = sc.kstar;
            R.n_fetch = wcnt[1];
        }
    }
    }
    stamp(5);

    cl.sync();   // no CTA leaves while its shared memory may still be read
    if (rank == 0 && tid == 0) {
        atomicAdd(a.dprog, 1ull);
        tline_stamp(a.tline, 8, false);
    }   // this row is decided (read by the prefetch)
}

// --------------------------------------------------------------------------------------------
// D7: union over the query heads of a KV head of L_g[:k*] \ S (per-row bitmaps set by the decision
// kernels), compacted to ascending tokens together with the mask of the query heads whose exact set
// holds each token (bit g); the bitmaps are cleared for the next call.  The rows themselves cross the
// host link inside the attention kernel, straight into its shared-memory ring.
// --------------------------------------------------------------------------------------------
// Weight factors of the sampled entries on the full-row path (the fused decision kernel writes
// them itself): 1 when the entry was made exact, lambda_i / r_i otherwise.
__global__ void __launch_bounds__(256) om_sampled_kernel(Views views, DecodeArgs a, const RowState* __restrict__ rows,
                                                         const float* __restrict__ wl, const int32_t* __restrict__ mark)
{
    const int row = blockIdx.y;
    const int b = row / a.Hq, kv = (row % a.Hq) / a.G;
    const SlotView& V = views.v[b];
    const int nl = rows[row].n_l;
    const float beta = rows[row].beta_f;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < nl; j += gridDim.x * blockDim.x) {
        const int sl = V.lslot[(int64_t)kv * V.n + j];
        if (sl < 0) continue;
        float w = 1.0f;
        if (mark[(int64_t)row * a.ws_n + j] != a.gen) {
            const float r = V.rl[(int64_t)kv * V.n + j];
            w = __fdiv_rn(lambda_of(wl[(int64_t)row * a.ws_n + j], r, beta), r);
        }
        a.om[(int64_t)row * a.ws_n + sl] = w;
    }
}

// --------------------------------------------------------------------------------------------
// Speculative prefetch (no counterpart in the algorithms; results are identical with it on or off).
// The host link idles while the decision runs, and the rows a decode ends up fetching are mostly the
// tokens of L \ S with the largest alpha = w^ (1 - r).  This kernel runs beside the decision (launched
// after it with programmatic dependent launch): per (sequence, KV head) it takes the tokens of
// L \ S that are neither sampled nor staged, keyed by their largest alpha over the head's query rows
// relative to each row's largest weight, log(alpha / w^_max) = max_g (t^_g - m_g) + log(1 - r); each of its blocks
// bins its share of them in steps of 1/16 over (-255/16, 0] (one read of the logits; the bins are kept
// in shared memory when the share fits), keeps the top pf_cap / gridDim.y by those bins and copies
// their K/V rows from pinned host memory into the call's prefetch buffer (a warp per row, 16 bytes a
// lane), recording token -> row.  Once every query row of the call is decided (the decision counts
// its rows) it stops: in the binning pass, before claiming rows and between the copies.  Before
// exiting it waits for the decision to complete, so that the attention, launched after it, sees
// both.  The attention reads a needed row from this buffer instead of the host when the buffer holds
// it.
// --------------------------------------------------------------------------------------------
constexpr int kPfThreads = 256;
constexpr int kPfBins = 255;         // bin 255 marks an entry that is not a candidate
constexpr int kPfListCap = 2048;     // candidates a prefetch block keeps
constexpr int kPfMaxRows = 4096;     // query rows of a call up to which the prefetch runs
constexpr int kPfShareCap = 32768;   // entries per block whose bins are kept in shared memory

// every query row of the call decided (the decision adds one per row to the counter, tagged with
// the call's generation)
__device__ __forceinline__ bool decision_done(const DecodeArgs& a, int rows_in_call)
{
    const unsigned long long p = *reinterpret_cast<volatile unsigned long long*>(a.dprog);
    return (unsigned)(p >> 32) == (unsigned)a.gen && (int)(p & 0xffffffffu) >= rows_in_call;
}

template <typename T, int G>
__global__ void __launch_bounds__(kPfThreads) prefetch_kernel(Views views, DecodeArgs a, const RowState* rows,
                                                              const float2* tl, int rows_in_call)
{
    constexpr int ROWB = 2 * kHeadDim * (int)sizeof(T);
    constexpr int CHUNKS = ROWB / 16;
    constexpr int U = 4;   // entries per thread in flight
    constexpr int NW = kPfThreads / 32;
    // host rows a warp reads at a time: two keep the link busy; more outstanding host reads slowed a
    // concurrent streaming decision by a quarter (batch 8 x 32K: 435 -> 540 us; with two, 445 us)
    constexpr int RF = 2;
    __shared__ unsigned hist[kPfBins], off[kPfBins];
    __shared__ int lst[kPfListCap];                 // candidates (L indices), then their tokens in bin order
    __shared__ unsigned char lbin[kPfListCap];
    __shared__ int s_n, s_thr, s_base, s_stop;
    extern __shared__ unsigned char sbin[];         // the share's bins (when it fits kPfShareCap)
    pdl_trigger();   // the attention may launch and wait at its own dependency point
    if (threadIdx.x == 0) tline_stamp(a.tline, 2, true);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int unit = blockIdx.x, b = unit / a.Hkv, kv = unit % a.Hkv;
    const SlotView& V = views.v[b];
    const int nl = V.counts[kv * 4 + 1];
    const int row0 = row_of(b, kv * G, a.Hq);
    const int per = (nl + gridDim.y - 1) / gridDim.y;
    const int j0 = min(nl, (int)blockIdx.y * per), j1 = min(nl, j0 + per);
    const int cap_blk = min(kPfListCap, a.pf_cap / (int)gridDim.y);
    const int64_t kvn = (int64_t)kv * V.n;
    const int32_t* stg_of = V.stage_of ? V.stage_of + kvn : nullptr;
    float m[G];
#pragma unroll
    for (int g = 0; g < G; ++g) m[g] = untag_max(__ldcg(&rows[row0 + g].m_tag), (unsigned)a.gen);
    // bins of U entries j = base + u T + tid (-1: sampled, so resident, or below the range); every load
    // of the group is issued before any is used
    auto bins = [&](int base, int (&bn)[U]) {
        int sl[U];
        float k[U], r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = base + u * kPfThreads + tid;
            sl[u] = j < j1 ? __ldg(V.lslot + kvn + j) : 0;
            r[u] = j < j1 ? __ldg(V.rl + kvn + j) : 0.f;
            k[u] = -INFINITY;
#pragma unroll
            for (int g = 0; g < G; ++g)
                if (j < j1) k[u] = fmaxf(k[u], __ldcg(tl + (int64_t)(row0 + g) * a.ws_n + j).x - m[g]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float kk = k[u] + __logf(1.0f - r[u]);   // log of alpha = w^ (1 - r) over the row's largest w^
            bn[u] = (sl[u] < 0 && kk > -(float)kPfBins / 16.0f) ? min(kPfBins - 1, (int)(-kk * 16.0f)) : -1;
        }
    };
    unsigned dyn_bytes;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
    const bool keep = j1 - j0 <= (int)dyn_bytes;   // the launch sized sbin for the largest share, or 0
    for (int i = tid; i < kPfBins; i += kPfThreads) hist[i] = 0u;
    if (tid == 0) {
        s_n = 0;
        s_stop = 0;
    }
    __syncthreads();
    // pass 1: the histogram of the block's share (a warp leaves it once the decision is complete)
    {
        int it = 0;
        for (int base = j0; base < j1; base += U * kPfThreads, ++it) {
            if ((it & 3) == 3) {
                bool dn = lane == 0 && decision_done(a, rows_in_call);
                dn = __shfl_sync(0xffffffffu, dn, 0);
                if (dn) {
                    if (lane == 0) s_stop = 1;
                    break;
                }
            }
            int bn[U];
            bins(base, bn);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (bn[u] >= 0) atomicAdd(&hist[bn[u]], 1u);
                const int j = base + u * kPfThreads + tid;
                if (keep && j < j1) sbin[j - j0] = (unsigned char)(bn[u] >= 0 ? bn[u] : kPfBins);
            }
        }
    }
    __syncthreads();
    if (tid == 0) tline_stamp(a.tline, 9, false);
    if (s_stop) {
        if (tid == 0) tline_stamp(a.tline, 10, false);
        pdl_wait();
        return;
    }
    if (warp == 0) {
        // the bins holding the block's top cap_blk (staged tokens are counted here and dropped below):
        // up to the first bin at which the running count reaches cap_blk, else all of them
        unsigned c[8], tot = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            c[j] = 8 * lane + j < kPfBins ? hist[8 * lane + j] : 0u;
            tot += c[j];
        }
        unsigned inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        int thr = -1;
        if (inc >= (unsigned)cap_blk && inc - tot < (unsigned)cap_blk) {
            unsigned cum = inc - tot;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                cum += c[j];
                if (thr < 0 && cum >= (unsigned)cap_blk) thr = 8 * lane + j;
            }
        }
        thr = __reduce_max_sync(0xffffffffu, thr);
        if (lane == 0) s_thr = thr >= 0 ? thr : kPfBins - 1;
    }
    __syncthreads();
    const int thr = s_thr;
    if (thr >= 0) {
        // pass 2: the candidates (at most cap_blk), then ordered by bin (a counting sort)
        auto take = [&](int j, int bn) {
            if (bn <= thr) {
                const int at = atomicAdd(&s_n, 1);
                if (at < cap_blk) {
                    lst[at] = j;
                    lbin[at] = (unsigned char)bn;
                }
            }
        };
        if (keep) {
            for (int i = tid; i < j1 - j0; i += kPfThreads) take(j0 + i, sbin[i]);
        } else {
            for (int base = j0; base < j1; base += U * kPfThreads) {
                int bn[U];
                bins(base, bn);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (bn[u] >= 0) take(base + u * kPfThreads + tid, bn[u]);
            }
        }
        __syncthreads();
        const int n0 = min(s_n, cap_blk);
        // their tokens; staged ones are dropped (-1): they are read from the staging cache anyway
        for (int i = tid; i < n0; i += kPfThreads) {
            const int tok = __ldg(V.ltok + kvn + lst[i]);
            lst[i] = (stg_of && __ldcg(stg_of + tok) >= 0) ? -1 : tok;
        }
        for (int i = tid; i < kPfBins; i += kPfThreads) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < n0; i += kPfThreads)
            if (lst[i] >= 0) atomicAdd(&hist[lbin[i]], 1u);
        __syncthreads();
        if (warp == 0) {
            // exclusive prefix of the kept counts over the bins (lane l: bins 8 l .. 8 l + 7)
            unsigned c[8], tot = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = 8 * lane + j < kPfBins ? hist[8 * lane + j] : 0u;
                tot += c[j];
            }
            unsigned inc = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            unsigned run = inc - tot;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (8 * lane + j < kPfBins) off[8 * lane + j] = run;
                run += c[j];
            }
            if (lane == 31) s_n = (int)inc;   // the kept candidates
        }
        __syncthreads();
        // the kept tokens in bin order (a counting sort through registers)
        int tk[kPfListCap / kPfThreads], ps[kPfListCap / kPfThreads];
#pragma unroll
        for (int u = 0; u < kPfListCap / kPfThreads; ++u) {
            const int i = u * kPfThreads + tid;
            tk[u] = i < n0 ? lst[i] : -1;
            ps[u] = tk[u] >= 0 ? (int)atomicAdd(&off[lbin[i]], 1u) : 0;
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kPfListCap / kPfThreads; ++u)
            if (tk[u] >= 0) lst[ps[u]] = tk[u];
        __syncthreads();
        const int n1 = s_n;
        if (tid == 0) s_base = atomicAdd(&a.pf_cnt[unit], n1);   // prefetch rows s_base .. of this block
        __syncthreads();
        const int base_row = s_base;
        unsigned char* buf = a.pf_buf + (int64_t)unit * a.pf_cap * ROWB;
        const unsigned char* host = reinterpret_cast<const unsigned char*>(V.kv_host) + kvn * ROWB;
        int32_t* pf_tok = a.pf_tok + (int64_t)unit * a.pf_cap;
        int32_t* pf_of = a.pf_of + (int64_t)unit * a.ws_n;
        // copies in bin order, a warp per row and two rows in flight (lane l moves bytes 16 l .. 16 l +
        // 15, and the next 512 when rows are fp32); once every query row of the call is decided the
        // remaining claimed rows are released (token -1), so the fetch no longer waits for them
        bool stop = false;
        for (int q0 = warp * RF; q0 < n1; q0 += RF * NW) {
            if (!stop && lane == 0) stop = decision_done(a, rows_in_call);
            stop = __shfl_sync(0xffffffffu, stop, 0);
            uint4 v[RF][CHUNKS / 32];
            int tok4[RF];
#pragma unroll
            for (int u = 0; u < RF; ++u) {
                const int qi = q0 + u;
                tok4[u] = qi < n1 && base_row + qi < a.pf_cap ? lst[qi] : -1;
                if (tok4[u] >= 0 && !stop) {
                    const uint4* src = reinterpret_cast<const uint4*>(host + (int64_t)tok4[u] * ROWB);
#pragma unroll
                    for (int c = 0; c < CHUNKS / 32; ++c) v[u][c] = __ldcs(src + lane + 32 * c);
                }
            }
#pragma unroll
            for (int u = 0; u < RF; ++u) {
                if (tok4[u] < 0) continue;
                const int sr = base_row + q0 + u;
                if (!stop) {
                    uint4* dst = reinterpret_cast<uint4*>(buf + (int64_t)sr * ROWB);
#pragma unroll
                    for (int c = 0; c < CHUNKS / 32; ++c) __stcs(dst + lane + 32 * c, v[u][c]);
                }
                if (lane == 0) {
                    pf_tok[sr] = stop ? -1 : tok4[u];
                    if (!stop) pf_of[tok4[u]] = sr;
                }
            }
        }
    }
    if (tid == 0) tline_stamp(a.tline, 10, false);
    pdl_wait();   // the decision has completed: the attention, launched after this grid, may read its results
}

// --------------------------------------------------------------------------------------------
// D8 (with the D7 copy): weighted attention (comment closing Algorithm 2; estimator of Theorem 2).
// Rows: the resident H u S rows of the KV head, then its fetched rows.  Per query head the weight
// factor is the one the scoring and decision kernels wrote for each resident slot (1 on H and on
// L_g[:k*], lambda_i / r_i on S \ L_g[:k*]) and, on a fetched row, 1 if the head's exact set holds
// it, else 0.  Each block takes every gridDim.y-th chunk of 32 KB of rows (64 bf16 rows) of one KV
// head into a two-stage shared-memory ring: a chunk of resident rows by one bulk asynchronous copy
// completed on an mbarrier, a chunk holding fetched rows by 16-byte cp.async copies whose sources
// for the fetched rows are the pinned host cache itself, so the host-link transfer overlaps the
// compute of the previous chunks and the rows never round-trip through HBM.  Per chunk: q.k for
// all G query heads (a row's 128 channels split over 2G threads), an online softmax per head, and
// p.v with two channels per thread; the last block of the KV head merges the splits.
// --------------------------------------------------------------------------------------------
constexpr int kAttnChunkBytes = 32768;
constexpr int kAttnStages = 2;
constexpr int kAttnThreads = 256;
constexpr int kMaxSplit = 128;              // attention splits per KV head (partials merged per query row)
template <typename T, int G>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_kernel(Views views, const float* __restrict__ q, DecodeArgs a,
                                                            const RowState* rows,
                                                            int32_t* __restrict__ ucount, int32_t* __restrict__ ulist,
                                                            uint8_t* __restrict__ umask, float* __restrict__ part,
                                                            int* __restrict__ done, float* __restrict__ out)
{
    constexpr int ROWB = 2 * kHeadDim * (int)sizeof(T);   // one K/V row
    constexpr int CR = kAttnChunkBytes / ROWB;             // rows per chunk
    constexpr int NS = kAttnStages;
    constexpr int QS = 64 / G;                             // channels per q.k thread
    constexpr int NSL = kHeadDim / QS;                     // threads per row in q.k (2G)
    constexpr int RSTEP = kAttnThreads / NSL;              // rows per q.k pass
    constexpr int EPT = (CR * G + kAttnThreads - 1) / kAttnThreads;  // weight factors per thread
    constexpr int PVI = (G * (kHeadDim / 2) + kAttnThreads - 1) / kAttnThreads;  // p.v items per thread
    static_assert(QS % 8 == 0 && CR <= 64 && CR >= 32, "attention tiling");
    extern __shared__ __align__(128) unsigned char sbuf[];  // NS x kAttnChunkBytes
    __shared__ __align__(8) unsigned long long full[NS];
    __shared__ float s_om[2][CR][G];
    __shared__ float s_p[CR][G];
    __shared__ float s_corr[G], s_m[G], s_l[G];
    __shared__ int s_bad;
    __shared__ int s_scan[32];
    __shared__ int s_sdst[NS][CR];   // staging-cache row to fill from a fetched row of the chunk (-1: none)
    __shared__ int s_stok[NS][CR];   // its token
    __shared__ int s_hcnt;           // rows this block read over the host link
    __shared__ int s_pcnt;           // rows this block read from the call's prefetch buffer
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int unit = blockIdx.x, b = unit / a.Hkv, kv = unit % a.Hkv;
    const SlotView& V = views.v[b];
    // resident rows: H u S of the compress (weights from om), then the appended tokens (weight 1)
    const int m_cmp = V.counts[kv * 4 + 3];
    const int m_res = m_cmp + V.n_tail;
    const int row0 = row_of(b, kv * G, a.Hq);   // the G query rows of the KV head are consecutive
    int32_t* ulw = ulist + (int64_t)unit * a.ws_n;
    uint8_t* umw = umask + (int64_t)unit * a.ws_n;
    // D7: the fetched rows of the KV head are the union of its G rows' L_g[:k*] \ S bitmaps, in
    // ascending tokens (no scan when none of the G rows fetches).  Every block counts all the words (thread t a contiguous run); the positions
    // of its own share below are written, with the mask of the heads holding each token, into the
    // fetch list, which the chunk copies read back.  Block 0 writes the count.
    // q slice of this thread (pre-scaled by 1/sqrt(d)), all G heads
    const int sl = tid % NSL;
    float qr[G][QS];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < QS; ++c) qr[g][c] = q[(int64_t)(row0 + g) * kHeadDim + sl * QS + c] * a.inv_sqrt_d_f;

    int nu = 0;
    pdl_wait();   // the decision kernel's bitmaps and weight factors are complete (the query is an input)
    if (tid == 0) tline_stamp(a.tline, 3, true);
    // the bitmaps are scanned only when a query row of the KV head fetches.  The counts come from the
    // decision kernel, which may still have been running when this grid started (programmatic launch):
    // they are read through L2, never through the non-coherent read-only path.
    int any_fetch = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) any_fetch |= __ldcg(&rows[row0 + g].n_fetch);
    if (!any_fetch) {
        if (blockIdx.y == 0 && tid == 0) ucount[unit] = 0;
    } else {
        const int64_t stride = a.ws_n / 32 + 1;
        const uint32_t* eb = a.ebits + (int64_t)row0 * stride;
        const int nwords = (V.n + 31) / 32;
        const int wpt = (nwords + kAttnThreads - 1) / kAttnThreads;
        const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
        int c = 0;
        for (int wi = w0; wi < w1; ++wi) {
            uint32_t wd = 0u;
#pragma unroll
            for (int g = 0; g < G; ++g) wd |= eb[g * stride + wi];
            c += __popc(wd);
        }
        const int pre = block_exclusive_scan(c, s_scan, &nu);
        const int pf_ = (nu + gridDim.y - 1) / gridDim.y;
        const int s0 = min(nu, (int)blockIdx.y * pf_), s1 = min(nu, s0 + pf_);
        if (c > 0 && pre < s1 && pre + c > s0) {
            int pos = pre;
            for (int wi = w0; wi < w1 && pos < s1; ++wi) {
                uint32_t wg[G];
                uint32_t wd = 0u;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    wg[g] = eb[g * stride + wi];
                    wd |= wg[g];
                }
                while (wd) {
                    const int bit = __ffs(wd) - 1;
                    if (pos >= s0 && pos < s1) {
                        unsigned m = 0u;
#pragma unroll
                        for (int g = 0; g < G; ++g) m |= ((wg[g] >> bit) & 1u) << g;
                        ulw[pos] = wi * 32 + bit;
                        umw[pos] = (uint8_t)m;
                    }
                    ++pos;
                    wd &= wd - 1u;
                }
            }
        }
        if (blockIdx.y == 0 && tid == 0) ucount[unit] = nu;
        __syncthreads();   // this block's share of the list is in place
    }
    // this block's rows: an equal share of the fetched rows (so that every block keeps the same
    // number of bytes on the host link) then an equal share of the resident rows; its chunks are
    // the fetched ones first, each chunk wholly fetched or wholly resident
    const int y = blockIdx.y, ny = gridDim.y;
    const int pf = (nu + ny - 1) / ny, pr = (m_res + ny - 1) / ny;
    const int f0 = min(nu, y * pf), nF = min(nu, f0 + pf) - f0;
    const int q0 = min(m_res, y * pr), nR = min(m_res, q0 + pr) - q0;
    const int nFc = (nF + CR - 1) / CR;
    const int nmine = nFc + (nR + CR - 1) / CR;
    // first row (index into resident rows, then fetched rows) and row count of chunk k
    auto chunk = [&](int k, int& r0, int& cnt) {
        if (k < nFc) {
            r0 = m_res + f0 + k * CR;
            cnt = min(CR, nF - k * CR);
        } else {
            r0 = q0 + (k - nFc) * CR;
            cnt = min(CR, nR - (k - nFc) * CR);
        }
    };
    const unsigned char* res = reinterpret_cast<const unsigned char*>(V.kvres) + V.res_off[kv] * (int64_t)ROWB;
    const unsigned char* host = reinterpret_cast<const unsigned char*>(V.kv_host) + (int64_t)kv * V.n * ROWB;
    const int32_t* ul = ulw;
    const uint8_t* um = umw;
    // the staging cache of the KV head: token -> staged row, the rows, their capacity
    int32_t* stg_of = V.stage_of ? V.stage_of + (int64_t)kv * V.n : nullptr;
    unsigned char* stg = stg_of ? reinterpret_cast<unsigned char*>(V.stage) + V.stage_off[kv] * (int64_t)ROWB : nullptr;
    const int stg_cap = stg_of ? (int)(V.stage_off[kv + 1] - V.stage_off[kv]) : 0;
    // the rows this call's prefetch copied ahead (written by the previous grid: read through L2)
    const int pf_n = a.pf_cap > 0 ? min(a.pf_cap, __ldcg(&a.pf_cnt[unit])) : 0;
    const int32_t* pf_of = a.pf_of + (int64_t)unit * a.ws_n;
    const int32_t* pf_tok = a.pf_tok + (int64_t)unit * a.pf_cap;
    const unsigned char* pfb = a.pf_buf + (int64_t)unit * a.pf_cap * ROWB;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_bad = 0;
        s_hcnt = 0;
        s_pcnt = 0;
    }
    if (tid < G) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    __syncthreads();

    // tokens of the fetched rows of chunk k and their staged rows: lane l < CR / 8 of warp w holds
    // those of row w + 8 l (staged row -1: not staged)
    auto load_tok = [&](int k) -> int2 {
        if (k >= nFc) return make_int2(0, -1);
        int r0, cnt;
        chunk(k, r0, cnt);
        const int row = warp + 8 * lane;
        if (!(lane < CR / 8 && row < cnt)) return make_int2(0, -1);
        const int tok = ul[r0 + row - m_res];
        int src = stg_of ? stg_of[tok] : -1;   // >= 0: staged row
        if (src < 0 && pf_n > 0) {
            // copied ahead by this call's prefetch: the row records it when its token agrees
            const int s = __ldcg(pf_of + tok);
            if (s >= 0 && s < pf_n && __ldcg(pf_tok + s) == tok) src = -2 - s;
        }
        return make_int2(tok, src);   // -1: read over the host link
    };
    // chunk k into stage k % NS.  A chunk of resident rows only is one bulk copy (thread 0); a chunk
    // holding fetched rows is copied 16 bytes per lane with cp.async, one row per warp at a time, the
    // fetched rows straight from the pinned host cache over the host link.  Every thread commits one
    // copy group per call (empty when k is past the block's chunks) so that the group count stays in
    // step with the chunk count; the stage's mbarrier completes one phase per chunk either way.
    // A fetched row that is staged is read from the staging cache in device memory; one that is not
    // crosses the host link and, while the cache has room, gets a staging row (filled once the chunk
    // has landed).
    auto issue = [&](int k, int2 tokreg) {
        if (k < nmine) {
            const int st = k % NS;
            int r0, cnt;
            chunk(k, r0, cnt);
            const int r1 = r0 + cnt;
            unsigned char* dst = sbuf + st * kAttnChunkBytes;
            if (k >= nFc) {
                if (tid == 0) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(&full[st], (unsigned)((r1 - r0) * ROWB));
                    bulk_g2s(dst, res + (int64_t)r0 * ROWB, (unsigned)((r1 - r0) * ROWB), &full[st]);
                }
            } else {
                if (tid == 0) mbar_arrive(&full[st]);
                const int myrow = warp + 8 * lane;
                if (lane < CR / 8) {
                    int sd = -1;
                    if (myrow < cnt && tokreg.y < 0) {
                        atomicAdd(tokreg.y == -1 ? &s_hcnt : &s_pcnt, 1);
                        if (stg_of) {
                            const int s_new = atomicAdd(&V.stage_cnt[kv], 1);
                            sd = s_new < stg_cap ? s_new : -1;
                        }
                    }
                    s_sdst[st][myrow] = sd;
                    s_stok[st][myrow] = tokreg.x;
                }
#pragma unroll
                for (int u = 0; u < CR / 8; ++u) {
                    const int row = warp + 8 * u, R = r0 + row;
                    const int tok = __shfl_sync(0xffffffffu, tokreg.x, u);
                    const int sidx = __shfl_sync(0xffffffffu, tokreg.y, u);
                    if (R < r1) {
                        const unsigned char* src = R < m_res   ? res + (int64_t)R * ROWB
                                                   : sidx >= 0  ? stg + (int64_t)sidx * ROWB
                                                   : sidx <= -2 ? pfb + (int64_t)(-2 - sidx) * ROWB
                                                                : host + (int64_t)tok * ROWB;
#pragma unroll
                        for (int p = lane; p < ROWB / 16; p += 32) cp_async16(dst + row * ROWB + p * 16, src + p * 16);
                    }
                }
            }
        }
        cp_async_commit();
    };
    // weight factors of chunk k, element e = r G + g of the chunk
    auto load_om = [&](int k, float (&o)[EPT]) {
        int r0, cnt;
        chunk(k, r0, cnt);
        const int r1 = r0 + cnt;
#pragma unroll
        for (int u = 0; u < EPT; ++u) {
            const int e = tid + u * kAttnThreads;
            const int r = e / G, g = e % G, R = r0 + r;
            float w = 0.f;
            if (e < CR * G && R < r1)
                w = R < m_cmp   ? a.om[(int64_t)(row0 + g) * a.ws_n + R]
                    : R < m_res ? 1.f
                                : (float)((um[R - m_res] >> g) & 1u);
            o[u] = w;
        }
    };
    auto store_om = [&](int buf, const float (&o)[EPT]) {
#pragma unroll
        for (int u = 0; u < EPT; ++u) {
            const int e = tid + u * kAttnThreads;
            if (e < CR * G) s_om[buf][e / G][e % G] = o[u];
        }
    };

    {
        int2 tk[NS];
#pragma unroll
        for (int k = 0; k < NS; ++k) tk[k] = load_tok(k);
#pragma unroll
        for (int k = 0; k < NS; ++k) issue(k, tk[k]);
    }
    float omv[EPT];
    if (nmine > 0) {
        load_om(0, omv);
        store_om(0, omv);
    }
    float acc[PVI][2];
#pragma unroll
    for (int u = 0; u < PVI; ++u) acc[u][0] = acc[u][1] = 0.f;

    int k = 0;
    for (; k < nmine; ++k) {
        const int st = k % NS;
        int r0, cnt;
        chunk(k, r0, cnt);
        if (k + 1 < nmine) load_om(k + 1, omv);   // stored at the end of this iteration
        const int2 tnext = load_tok(k + NS);        // used when chunk k + NS is issued below
        __syncthreads();
        if (!mbar_wait(&full[st], (unsigned)((k / NS) & 1), kWaitLimit)) atomicOr(&s_bad, 1);
        cp_async_wait<NS - 1>();                    // this thread's copies of chunk k have landed
        __syncthreads();
        if (s_bad) break;
        const unsigned char* buf = sbuf + st * kAttnChunkBytes;
        if (k < nFc && stg_of) {
            // fill the staging rows given to this chunk's newly fetched rows (warp w: rows w + 8 u)
#pragma unroll
            for (int u = 0; u < CR / 8; ++u) {
                const int row = warp + 8 * u;
                const int sd = s_sdst[st][row];
                if (row < cnt && sd >= 0) {
                    unsigned char* drow = stg + (int64_t)sd * ROWB;
#pragma unroll
                    for (int p = lane; p < ROWB / 16; p += 32)
                        *reinterpret_cast<uint4*>(drow + p * 16) = *reinterpret_cast<const uint4*>(buf + row * ROWB + p * 16);
                    if (lane == 0) stg_of[s_stok[st][row]] = sd;
                }
            }
        }
        // q.k: thread (row, slice); the 2G threads of a row are consecutive lanes
        for (int r = tid / NSL; r < CR; r += RSTEP) {
            float d[G];
#pragma unroll
            for (int g = 0; g < G; ++g) d[g] = 0.f;
            if (r < cnt) {
                const unsigned char* kr = buf + r * ROWB + sl * QS * (int)sizeof(T);
#pragma unroll
                for (int c8 = 0; c8 < QS; c8 += 8) {
                    float kk[8];
                    RowCvt<T>::load8(kr + c8 * (int)sizeof(T), kk);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int c = 0; c < 8; ++c) d[g] = fmaf(qr[g][c8 + c], kk[c], d[g]);
                }
            }
#pragma unroll
            for (int o = 1; o < NSL; o <<= 1)
#pragma unroll
                for (int g = 0; g < G; ++g) d[g] += __shfl_xor_sync(0xffffffffu, d[g], o);
            if (sl < G) {
                float x = d[0];
#pragma unroll
                for (int g = 1; g < G; ++g)
                    if (sl == g) x = d[g];
                s_p[r][sl] = (r < cnt && s_om[k & 1][r][sl] > 0.f) ? x : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax: warp g takes query head g
        if (warp < G) {
            const int g = warp;
            float x[CR / 32], p[CR / 32];
            float cmax = -INFINITY;
#pragma unroll
            for (int h = 0; h < CR / 32; ++h) {
                x[h] = s_p[lane + 32 * h][g];
                cmax = fmaxf(cmax, x[h]);
            }
            cmax = warp_max(cmax);
            const float Mold = s_m[g], Mnew = fmaxf(Mold, cmax);
            float corr = 1.f, ls = 0.f;
            if (Mnew > -INFINITY) {
                corr = Mold > -INFINITY ? expf(Mold - Mnew) : 0.f;
#pragma unroll
                for (int h = 0; h < CR / 32; ++h) {
                    p[h] = x[h] > -INFINITY ? s_om[k & 1][lane + 32 * h][g] * expf(x[h] - Mnew) : 0.f;
                    ls += p[h];
                }
            } else {
#pragma unroll
                for (int h = 0; h < CR / 32; ++h) p[h] = 0.f;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
#pragma unroll
            for (int h = 0; h < CR / 32; ++h) s_p[lane + 32 * h][g] = p[h];
            __syncwarp();
            if (lane == 0) {
                s_l[g] = s_l[g] * corr + ls;
                s_m[g] = Mnew;
                s_corr[g] = corr;
            }
        }
        __syncthreads();
        // p.v: item (g, channel pair)
#pragma unroll
        for (int u = 0; u < PVI; ++u) {
            const int e = tid + u * kAttnThreads;
            if (e < G * (kHeadDim / 2)) {
                const int g = e / (kHeadDim / 2), c2 = 2 * (e % (kHeadDim / 2));
                const float cr = s_corr[g];
                float a0 = acc[u][0] * cr, a1 = acc[u][1] * cr;
                const unsigned char* vb = buf + kHeadDim * (int)sizeof(T) + c2 * (int)sizeof(T);
                for (int r = 0; r < cnt; ++r) {
                    const float pr = s_p[r][g];
                    const float2 v = RowCvt<T>::load2(vb + r * ROWB);
                    a0 = fmaf(pr, v.x, a0);
                    a1 = fmaf(pr, v.y, a1);
                }
                acc[u][0] = a0;
                acc[u][1] = a1;
            }
        }
        if (k + 1 < nmine) store_om((k + 1) & 1, omv);
        __syncthreads();   // stage st and s_p are free
        issue(k + NS, tnext);
    }
    if (s_bad) {
        // a copy did not complete in time: report it, and before leaving wait (bounded) for the
        // copies this block still has in flight
        if (tid == 0) {
            *(volatile int*)a.err = 1;
            for (int kk = k; kk < min(nmine, k + NS); ++kk) mbar_wait(&full[kk % NS], (unsigned)((kk / NS) & 1), kWaitLimit);
        }
        cp_async_wait<0>();
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < PVI; ++u) {
        const int e = tid + u * kAttnThreads;
        if (e < G * (kHeadDim / 2)) {
            const int g = e / (kHeadDim / 2), c2 = 2 * (e % (kHeadDim / 2));
            float* pp = part + ((int64_t)(row0 + g) * a.nsplit + y) * (kHeadDim + 2);
            pp[c2] = acc[u][0];
            pp[c2 + 1] = acc[u][1];
            if (c2 == 0) {
                pp[kHeadDim] = s_m[g];
                pp[kHeadDim + 1] = s_l[g];
            }
        }
    }
    // the last block of the KV head to finish merges the gridDim.y partials of its G query rows
    // (log-sum-exp over the splits); the counter is left at zero for the next call
    if (tid == 0 && s_hcnt > 0) atomicAdd(&a.hrows[unit], s_hcnt);
    if (tid == 0 && s_pcnt > 0) atomicAdd(&a.pf_used[unit], s_pcnt);
    __shared__ int s_last;
    __shared__ float s_scl[G][kMaxSplit], s_lsp[G][kMaxSplit];
    __shared__ float s_L[G];
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&done[unit], 1) == ny - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // (m, l) of every split and head in one pass, then the scale factors, then the outputs
    for (int e = tid; e < G * ny; e += kAttnThreads) {
        const int g = e / ny, sp = e % ny;
        const float* pp = part + ((int64_t)(row0 + g) * a.nsplit + sp) * (kHeadDim + 2);
        s_scl[g][sp] = pp[kHeadDim];
        s_lsp[g][sp] = pp[kHeadDim + 1];
    }
    __syncthreads();
    if (warp < G) {
        const int g = warp;
        float M = -INFINITY;
        for (int sp = lane; sp < ny; sp += 32) M = fmaxf(M, s_scl[g][sp]);
        M = warp_max(M);
        float L = 0.f;
        for (int sp = lane; sp < ny; sp += 32) {
            const float m = s_scl[g][sp];
            const float f = m == -INFINITY ? 0.f : expf(m - M);
            s_scl[g][sp] = f;
            L += s_lsp[g][sp] * f;
        }
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) s_L[g] = L;
    }
    __syncthreads();
    for (int e = tid; e < G * kHeadDim; e += kAttnThreads) {
        const int g = e / kHeadDim, c = e % kHeadDim;
        const float* pr = part + (int64_t)(row0 + g) * a.nsplit * (kHeadDim + 2);
        float A0 = 0.f, A1 = 0.f, A2 = 0.f, A3 = 0.f;
        int sp = 0;
        for (; sp + 4 <= ny; sp += 4) {
            A0 = fmaf(pr[sp * (kHeadDim + 2) + c], s_scl[g][sp], A0);
            A1 = fmaf(pr[(sp + 1) * (kHeadDim + 2) + c], s_scl[g][sp + 1], A1);
            A2 = fmaf(pr[(sp + 2) * (kHeadDim + 2) + c], s_scl[g][sp + 2], A2);
            A3 = fmaf(pr[(sp + 3) * (kHeadDim + 2) + c], s_scl[g][sp + 3], A3);
        }
        for (; sp < ny; ++sp) A0 = fmaf(pr[sp * (kHeadDim + 2) + c], s_scl[g][sp], A0);
        out[(int64_t)(row0 + g) * kHeadDim + c] = ((A0 + A1) + (A2 + A3)) / s_L[g];
    }
    if (tid == 0) {
        done[unit] = 0;
        tline_stamp(a.tline, 11, false);
    }
}

int g_decide_max_cluster = 8;  // largest cluster the decide kernel is launched with (set once)

template <typename T, int G>
verkv_status launch_decode(Ctx& ctx, const Views& views, const DecodeArgs& a, int B, int max_n, int max_nl,
                           int max_nh, int max_res, const float* q, float* out, cudaStream_t st)
{
    const verkv_config& cfg = ctx.cfg;
    const int rowsN = B * a.Hq;
    VK_TIMING_BEGIN();
    // The fused decision takes rows of up to kDecideMaxL entries.  It keeps the entries in shared
    // memory (clusters of C CTAs of kDecideCap entries, one CTA per multiprocessor) when every row of
    // the call fits one wave; otherwise the streaming variant re-reads them from L2 in every pass, with
    // two CTAs per multiprocessor and clusters of Cs CTAs sized so the call's rows fill about one wave.
    int C = 1;
    while (C * kDecideCap < max_nl) C <<= 1;
    const bool on_chip = max_nl <= kDecideMaxL;
    const bool stream = on_chip && !(max_nl <= g_decide_max_cluster * kDecideCap && rowsN * C <= ctx.num_sms);
    int Cs = 1;
    while (Cs * 2 <= kDecideStreamMaxCluster && rowsN * Cs * 2 <= 2 * ctx.num_sms) Cs <<= 1;
    if (!on_chip) {
        init_rows_kernel<<<(rowsN + 127) / 128, 128, 0, st>>>(ctx.rows, views, a, B);
        VK_LAUNCHED("init_rows");
        // the fused decision kernel clears its row's exact-set bitmap itself; this path starts clean
        VK_CUDA(cudaMemsetAsync(a.ebits, 0, sizeof(uint32_t) * rowsN * (a.ws_n / 32 + 1), st));
    }
    // one launch scores L (sketch tiles) and H (exact tiles past them)
    const int h_tiles = (max_nh + kHTilesPerBlock * (kTile / (8 * G)) - 1) / (kHTilesPerBlock * (kTile / (8 * G)));
    if (cfg.sketch == VERKV_SKETCH_INT8) {
        static bool int8_attr = false;   // one per (T, G) instantiation
        if (!int8_attr) {
            VK_CUDA(cudaFuncSetAttribute(score_int8_kernel<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Int8Mma<G>::Smem));
            int8_attr = true;
        }
        // CTAs per (sequence, KV head): about kInt8CtasPerSm per multiprocessor over the call
        const int mt = (max_n + 127) / 128;
        const int lt = std::max(1, std::min(mt, kInt8CtasPerSm * ctx.num_sms / (B * a.Hkv)));   // one wave
        score_int8_kernel<T, G><<<dim3(lt, B * a.Hkv), kTile, Int8Mma<G>::Smem, st>>>(views, q, a, ctx.rows,
                                                                                               ctx.tl, ctx.th, lt);
    } else if (cfg.sketch == VERKV_SKETCH_2BIT) {
        const int lt = ((max_n + kTile - 1) / kTile + kGroupsPerBlock - 1) / kGroupsPerBlock;
        score_2bit_kernel<T, G><<<dim3(lt + h_tiles, B * a.Hkv), kTile, 0, st>>>(views, q, a, ctx.rows, ctx.tl, ctx.th, lt);
    } else {
        const int lt = (max_n + kTile - 1) / kTile;
        score_exact_kernel<T, G><<<dim3(lt + h_tiles, B * a.Hkv), kTile, 0, st>>>(views, q, a, ctx.rows, ctx.tl, ctx.th, lt);
    }
    VK_LAUNCHED("score");
    if (ctx.shortlist_k > 0) {
        // keys: about two blocks per multiprocessor over the call, at least 2048 entries a block
        const int units = B * a.Hkv;
        const int ny = std::max(1, std::min((max_nl + 4 * kSlThreads - 1) / (4 * kSlThreads),
                                            2 * ctx.num_sms / units));
        const int yb = ny + (max_res + kSlThreads / 4 - 1) / (kSlThreads / 4);   // four lanes per sampled key
        shortlist_keys_kernel<T, G><<<dim3(units, yb), kSlThreads, 0, st>>>(
            views, q, a, ctx.rows, ctx.tl, reinterpret_cast<unsigned*>(ctx.keys), ctx.shist, ny);
        VK_LAUNCHED("shortlist_keys");
        shortlist_select_kernel<T, G><<<units, kSlThreads, 0, st>>>(views, q, a, ctx.rows, ctx.tl, ctx.shortlist_k,
                                                                    ctx.slist, ctx.scount,
                                                                    reinterpret_cast<const unsigned*>(ctx.keys),
                                                                    ctx.shist);
        VK_LAUNCHED("shortlist");
    }
    if (on_chip) {
        const int CC = stream ? Cs : C;
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(rowsN * CC);
        lc.blockDim = dim3(stream ? kDecideStreamThreads : kDecideThreads);
        lc.dynamicSmemBytes = stream ? kDecideHistSmem : kDecideSmem;
        lc.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CC;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = attr;
        lc.numAttrs = 2;
        auto kern = a.binary ? (stream ? decide_kernel<true, true> : decide_kernel<true, false>)
                             : (stream ? decide_kernel<false, true> : decide_kernel<false, false>);
        VK_CUDA(cudaLaunchKernelEx(&lc, kern, views, a, ctx.rows, (const float2*)ctx.tl, (const float2*)ctx.th,
                                   ctx.wl, ctx.mark, ctx.elist, ctx.keys));
        VK_LAUNCHED("decide");
    } else {
        const int wmax = std::max(max_nl, max_nh);
        weights_kernel<<<dim3(std::max(1, (wmax + 255) / 256), rowsN), 256, 0, st>>>(views, a, ctx.rows, ctx.tl,
                                                                                    ctx.th, ctx.wl);
        VK_LAUNCHED("weights");
        beta_kernel<<<rowsN, 1024, 0, st>>>(views, a, ctx.rows, ctx.wl);
        VK_LAUNCHED("beta");
        const size_t sel_smem = sizeof(unsigned long long) * kSelWidth;
        select_kernel<<<rowsN, 1024, sel_smem, st>>>(views, a, ctx.rows, ctx.wl, ctx.keys, ctx.mark, ctx.elist);
        VK_LAUNCHED("select");
    }
    if (!on_chip) {
        fallback_kernel<<<rowsN, 1024, 0, st>>>(views, a, ctx.rows, ctx.wl, ctx.keys, ctx.mark, ctx.elist);
        VK_LAUNCHED("fallback");
    }
    if (!on_chip) {
        om_sampled_kernel<<<dim3(std::max(1, std::min(64, (max_nl + 255) / 256)), rowsN), 256, 0, st>>>(
            views, a, ctx.rows, ctx.wl, ctx.mark);
        VK_LAUNCHED("om_sampled");
    }
    // beside the decision: on the multiprocessors its CTAs leave free (one CTA per SM on chip, two
    // streaming), four prefetch blocks each, shared out over the call's (sequence, KV head) units (at
    // least one per unit).  Calls whose decision leaves fewer than eight multiprocessors free run
    // without it.
    const int dec_ctas = rowsN * (stream ? Cs : C);
    const int free_sms = std::max(0, ctx.num_sms - (stream ? (dec_ctas + 1) / 2 : dec_ctas));
    const bool prefetch = on_chip && a.pf_cap > 0 && rowsN <= kPfMaxRows && free_sms >= 8;
    ctx.last_pf_cap = prefetch ? a.pf_cap : 0;
    if (prefetch) {
        const int nb = std::max(1, std::min(16, 4 * free_sms / (B * a.Hkv)));
        const int share = (max_nl + nb - 1) / nb;
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(B * a.Hkv, nb);
        lc.blockDim = dim3(kPfThreads);
        lc.dynamicSmemBytes = share <= kPfShareCap ? (size_t)((share + 15) & ~15) : 0;
        lc.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        VK_CUDA(cudaLaunchKernelEx(&lc, prefetch_kernel<T, G>, views, a, (const RowState*)ctx.rows,
                                   (const float2*)ctx.tl, rowsN));
        VK_LAUNCHED("prefetch");
    }
    static bool attn_attr = false;   // one per (T, G) instantiation
    if (!attn_attr) {
        VK_CUDA(cudaFuncSetAttribute(attn_kernel<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kAttnStages * kAttnChunkBytes));
        attn_attr = true;
    }
    {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(B * a.Hkv, a.nsplit);
        lc.blockDim = dim3(kAttnThreads);
        lc.dynamicSmemBytes = kAttnStages * kAttnChunkBytes;
        lc.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        VK_CUDA(cudaLaunchKernelEx(&lc, attn_kernel<T, G>, views, q, a, (const RowState*)ctx.rows, ctx.ucount, ctx.ulist,
                                   ctx.umask, ctx.part,
                                   a.done, out));
    }
    VK_LAUNCHED("attn");
    return VERKV_OK;
}

template <typename T>
verkv_status dispatch_g(Ctx& ctx, const Views& views, const DecodeArgs& a, int B, int max_n, int max_nl, int max_nh,
                        int max_res, const float* q, float* out, cudaStream_t st)
{
    switch (ctx.G) {
        case 1: return launch_decode<T, 1>(ctx, views, a, B, max_n, max_nl, max_nh, max_res, q, out, st);
        case 2: return launch_decode<T, 2>(ctx, views, a, B, max_n, max_nl, max_nh, max_res, q, out, st);
        case 4: return launch_decode<T, 4>(ctx, views, a, B, max_n, max_nl, max_nh, max_res, q, out, st);
        case 8: return launch_decode<T, 8>(ctx, views, a, B, max_n, max_nl, max_nh, max_res, q, out, st);
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
        VK_CUDA(cudaFuncSetAttribute(decide_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecideSmem));
        VK_CUDA(cudaFuncSetAttribute(decide_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecideSmem));
        VK_CUDA(cudaFuncSetAttribute(decide_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kDecideHistSmem));
        VK_CUDA(cudaFuncSetAttribute(decide_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kDecideHistSmem));
        // a 16-CTA cluster (non-portable) lets rows of up to 16 x kDecideCap entries stay on chip
        if (cudaFuncSetAttribute(decide_kernel<false, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
            cudaFuncSetAttribute(decide_kernel<true, false>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(kDecideMaxCluster);
            lc.blockDim = dim3(kDecideThreads);
            lc.dynamicSmemBytes = kDecideSmem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = kDecideMaxCluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            lc.attrs = attr;
            lc.numAttrs = 1;
            int nclusters = 0;
            if (cudaOccupancyMaxActiveClusters(&nclusters, decide_kernel<false, false>, &lc) == cudaSuccess && nclusters > 0)
                g_decide_max_cluster = kDecideMaxCluster;
        }
        cudaGetLastError();  // a refused query leaves no error behind
        g_attr_done = true;
    }
    Views views;
    memset(&views, 0, sizeof(views));
    int max_n = 0, max_nl = 0, max_nh = 0, max_res = 0;
    ctx.last_seq.assign(seq_ids, seq_ids + B);
    ctx.last_n.clear();
    for (int b = 0; b < B; ++b) {
        Slot& s = ctx.slot(layer, seq_ids[b]);
        SlotView& v = views.v[b];
        v.n = s.n;
        v.n_tail = s.n_tail;
        v.r = s.r;
        v.flags = s.flags;
        v.lpos = s.lpos;
        v.ltok = s.ltok;
        v.rl = s.rl;
        v.lslot = s.lslot;
        v.lq = s.lq;
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
        const bool staged = !s.stage_off_host.empty() && s.stage_off_host.back() > 0;
        v.stage_of = staged ? s.stage_of : nullptr;
        v.stage = s.stage;
        v.stage_off = s.stage_off;
        v.stage_cnt = s.stage_cnt;
        max_n = std::max(max_n, s.n);
        for (const verkv_head_stats& hs : s.stats) {
            max_nl = std::max(max_nl, hs.n_l);
            max_nh = std::max(max_nh, hs.n_h + s.n_tail);
            max_res = std::max(max_res, hs.n_resident);
        }
        ctx.last_n.push_back(s.n);
    }
    if (cfg.shrinkage == VERKV_SHRINK_BINARY && max_nl > kDecideMaxL) {
        ctx.err = "binary shrinkage runs in the fused decision: |L| of a row is above 262144";
        return VERKV_EUNSUPPORTED;
    }
    DecodeArgs a;
    a.Hkv = cfg.n_kv_heads;
    a.binary = cfg.shrinkage == VERKV_SHRINK_BINARY ? 1 : 0;
    a.Hq = cfg.n_q_heads;
    a.G = ctx.G;
    a.ws_n = ctx.ws_n;
    a.ws_npow2 = ctx.ws_npow2;
    a.gen = ++ctx.gen;
    a.ebits = ctx.ebits;
    a.om = ctx.om;
    a.err = ctx.d_err;
    a.done = ctx.adone;
    a.hrows = ctx.hrows;
    if (ctx.prefetch_rows > 0 && ctx.pf_cap != ctx.prefetch_rows) {
        // the prefetch buffers, sized at the first decode after a change of the setting
        if (ctx.pf_buf) VK_CUDA(cudaFree(ctx.pf_buf));
        if (ctx.pf_tok) VK_CUDA(cudaFree(ctx.pf_tok));
        ctx.pf_buf = nullptr;
        ctx.pf_tok = nullptr;
        ctx.pf_cap = 0;
        const size_t kvb = (size_t)cfg.max_batch * cfg.n_kv_heads;
        VK_CUDA(cudaMalloc(&ctx.pf_buf, kvb * (size_t)ctx.prefetch_rows * 2 * kHeadDim * ctx.elt));
        VK_CUDA(cudaMalloc(&ctx.pf_tok, sizeof(int32_t) * kvb * (size_t)ctx.prefetch_rows));
        if (!ctx.pf_of) {
            VK_CUDA(cudaMalloc(&ctx.pf_of, sizeof(int32_t) * kvb * (size_t)ctx.ws_n));
            VK_CUDA(cudaMemsetAsync(ctx.pf_of, 0xff, sizeof(int32_t) * kvb * (size_t)ctx.ws_n, st));
        }
        ctx.pf_cap = ctx.prefetch_rows;
    }
    a.pf_cap = ctx.prefetch_rows > 0 ? ctx.pf_cap : 0;
    a.pf_buf = reinterpret_cast<unsigned char*>(ctx.pf_buf);
    a.pf_of = ctx.pf_of;
    a.pf_tok = ctx.pf_tok;
    a.pf_cnt = ctx.pf_cnt;
    a.pf_used = ctx.pf_used;
    a.dprog = ctx.dprog;
    a.tline = nullptr;
    if (ctx.timeline) {
        if (!ctx.tline) VK_CUDA(cudaMalloc(&ctx.tline, sizeof(unsigned long long) * 16));
        VK_CUDA(cudaMemsetAsync(ctx.tline, 0xff, sizeof(unsigned long long) * 8, st));
        VK_CUDA(cudaMemsetAsync(ctx.tline + 8, 0, sizeof(unsigned long long) * 8, st));
        a.tline = ctx.tline;
    }
    ctx.last_tline = ctx.timeline;
    // attention splits per KV head: about two blocks per SM over the whole call
    a.nsplit = std::min(std::min(ctx.nsplit, kMaxSplit), std::max(1, (2 * ctx.num_sms + B * cfg.n_kv_heads - 1) / (B * cfg.n_kv_heads)));
    a.eps = eps;
    a.eps_f = (float)eps;
    a.ldelta = std::log(2.0 / delta);
    a.eps_ff.hi = (float)eps;
    a.eps_ff.lo = (float)(eps - (double)a.eps_ff.hi);
    a.ld_ff.hi = (float)a.ldelta;
    a.ld_ff.lo = (float)(a.ldelta - (double)a.ld_ff.hi);
    const double isd = 1.0 / std::sqrt((double)kHeadDim);
    a.inv_sqrt_d_f = (float)isd;
    a.inv_sqrt_d.hi = (float)isd;
    a.inv_sqrt_d.lo = (float)(isd - (double)(float)isd);
    ctx.last_launches = 0;
    ctx.last_B = B;
    ctx.last_layer = layer;
    if (cfg.kv_dtype == VERKV_DTYPE_BF16)
        return dispatch_g<__nv_bfloat16>(ctx, views, a, B, max_n, max_nl, max_nh, max_res, q, out, st);
    return dispatch_g<float>(ctx, views, a, B, max_n, max_nl, max_nh, max_res, q, out, st);
}

}  // namespace verkv

// ================================================================================================
// Allocation-free variant of the per-row decision (the beta solve, the certificate, the gains, the
// full-row ranking and k* of the full-row path above) for callers that cannot allocate device memory: code
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
    // inputs outside the documented domain (r not in (0, 1), w negative or not finite) give k* = -1
    // and NaN scalars instead of a silent inf / NaN from the divisions below
    int bad = 0;
    for (int j = threadIdx.x; j < nl; j += blockDim.x) {
        const float wj = w[j], rj = rr[j];
        bad |= !(rj > 0.f && rj < 1.f) || !(wj >= 0.f && wj <= 3.4028234663852886e38f);
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) {
            for (int i = 0; i < 4; ++i) out_scalars[i] = __longlong_as_double(0x7ff8000000000000ll);
            *out_kstar = -1;
        }
        return;
    }
    if (nl == 0) {   // empty L: nothing to estimate, eps_hat = 0, and nothing to fetch whatever eps is
        if (threadIdx.x == 0) {
            for (int i = 0; i < 4; ++i) out_scalars[i] = 0.0;
            *out_kstar = 0;
        }
        return;
    }
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
    kstar = min(max(kstar, 1), nl);   // eps_hat(L) >= eps here, so k* >= 1; k = |L| is always accepted
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
