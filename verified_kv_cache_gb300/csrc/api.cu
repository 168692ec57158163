// C ABI of libverkv.so (declared in include/verkv.h): argument checks, slot bookkeeping, the
// decode workspace and the inspection getters.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "async.cuh"
#include "common.cuh"
#include "internal.h"

namespace verkv {
int decode_max_batch();
int decode_sel_width();
}  // namespace verkv

using namespace verkv;

struct verkv_ctx {
    Ctx c;
};

namespace {

verkv_status fail(Ctx& ctx, verkv_status s, const char* msg)
{
    ctx.err = msg;
    return s;
}

void free_ws(Ctx& c)
{
    void* ptrs[] = {c.tl, c.th, c.wl, c.rows, c.keys, c.mark, c.elist, c.ebits, c.om, c.ulist, c.umask, c.adone, c.ucount,
                    c.part, c.hrows, c.slist, c.scount, c.shist,
                    c.d_slot_n, c.pf_buf, c.pf_of, c.pf_tok, c.pf_cnt, c.pf_used, c.dprog, c.tau_ws, c.tline};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    if (c.h_err) cudaFreeHost(c.h_err);
}

verkv_status alloc_ws(Ctx& ctx)
{
    const verkv_config& cfg = ctx.cfg;
    const size_t rows = (size_t)cfg.max_batch * cfg.n_q_heads;
    const size_t n = (size_t)cfg.max_tokens;
    int p2 = 1;
    while (p2 < cfg.max_tokens) p2 <<= 1;
    ctx.ws_rows = (int)rows;
    ctx.ws_n = cfg.max_tokens;
    ctx.ws_npow2 = p2;
    const size_t kvb = (size_t)cfg.max_batch * cfg.n_kv_heads;
    VK_CUDA(cudaMalloc(&ctx.tl, sizeof(float2) * rows * n));
    VK_CUDA(cudaMalloc(&ctx.th, sizeof(float2) * rows * n));
    VK_CUDA(cudaMalloc(&ctx.wl, sizeof(float) * rows * n));
    VK_CUDA(cudaMalloc(&ctx.rows, sizeof(RowState) * rows));
    VK_CUDA(cudaMemset(ctx.rows, 0, sizeof(RowState) * rows));
    // at least two words a row: the shortlist reuses the buffer as rows of 2 max(p2, 2) 32-bit keys,
    // one per KV head, written four at a time
    VK_CUDA(cudaMalloc(&ctx.keys, sizeof(unsigned long long) * rows * (size_t)std::max(p2, 2)));
    VK_CUDA(cudaMalloc(&ctx.mark, sizeof(int32_t) * rows * n));
    VK_CUDA(cudaMemset(ctx.mark, 0, sizeof(int32_t) * rows * n));
    VK_CUDA(cudaMalloc(&ctx.elist, sizeof(int32_t) * rows * n));
    VK_CUDA(cudaMalloc(&ctx.ebits, sizeof(uint32_t) * rows * (n / 32 + 1)));
    VK_CUDA(cudaMemset(ctx.ebits, 0, sizeof(uint32_t) * rows * (n / 32 + 1)));
    VK_CUDA(cudaMalloc(&ctx.om, sizeof(float) * rows * n));
    VK_CUDA(cudaMalloc(&ctx.ulist, sizeof(int32_t) * kvb * n));
    VK_CUDA(cudaMalloc(&ctx.umask, kvb * n));
    VK_CUDA(cudaMalloc(&ctx.adone, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMemset(ctx.adone, 0, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMalloc(&ctx.ucount, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMemset(ctx.ucount, 0, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMalloc(&ctx.hrows, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMemset(ctx.hrows, 0, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMalloc(&ctx.pf_cnt, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMemset(ctx.pf_cnt, 0, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMalloc(&ctx.pf_used, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMemset(ctx.pf_used, 0, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMalloc(&ctx.dprog, sizeof(unsigned long long)));
    VK_CUDA(cudaMemset(ctx.dprog, 0, sizeof(unsigned long long)));
    VK_CUDA(cudaMalloc(&ctx.slist, sizeof(int32_t) * kvb * kMaxShortlist));
    VK_CUDA(cudaMalloc(&ctx.scount, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMemset(ctx.scount, 0, sizeof(int32_t) * kvb));
    VK_CUDA(cudaMalloc(&ctx.shist, sizeof(uint32_t) * kvb * (kShortlistBins + 1)));
    VK_CUDA(cudaMemset(ctx.shist, 0, sizeof(uint32_t) * kvb * (kShortlistBins + 1)));
    VK_CUDA(cudaMalloc(&ctx.part, sizeof(float) * rows * ctx.nsplit * (kHeadDim + 2)));
    VK_CUDA(cudaHostAlloc(reinterpret_cast<void**>(&ctx.h_err), sizeof(int), cudaHostAllocMapped));
    *ctx.h_err = 0;
    VK_CUDA(cudaHostGetDevicePointer(reinterpret_cast<void**>(&ctx.d_err), ctx.h_err, 0));
    return VERKV_OK;
}

// The mapped error word is written by a kernel whose bounded wait gave up; reading it clears it.
bool take_device_timeout(Ctx& ctx)
{
    if (!ctx.h_err || *reinterpret_cast<volatile int*>(ctx.h_err) == 0) return false;
    *reinterpret_cast<volatile int*>(ctx.h_err) = 0;
    return true;
}

bool slot_ok(const Ctx& c, int layer, int seq)
{
    return layer >= 0 && layer < c.cfg.n_layers && seq >= 0 && seq < c.cfg.n_seqs;
}

// One block waits on an mbarrier that nothing arrives at, with the bounded wait every kernel uses
// (a shorter limit), and raises the error word when it gives up.
__global__ void wait_timeout_kernel(int* err)
{
    __shared__ unsigned long long bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait(&bar, 0u, 1u << 14)) *(volatile int*)err = 1;
    }
}

}  // namespace

extern "C" {

const char* verkv_status_str(verkv_status s)
{
    switch (s) {
        case VERKV_OK: return "ok";
        case VERKV_EINVAL: return "invalid argument";
        case VERKV_ENOMEM: return "out of memory";
        case VERKV_ECUDA: return "CUDA error";
        case VERKV_ETIMEOUT: return "device wait timed out";
        case VERKV_EUNSUPPORTED: return "unsupported configuration";
        case VERKV_ESTATE: return "call out of order";
    }
    return "unknown status";
}

const char* verkv_last_error(const verkv_ctx* ctx) { return ctx ? ctx->c.err.c_str() : "null context"; }

int32_t verkv_last_launch_count(const verkv_ctx* ctx) { return ctx ? ctx->c.last_launches : 0; }

verkv_status verkv_create(const verkv_config* cfg, verkv_ctx** out)
{
    if (!cfg || !out) return VERKV_EINVAL;
    *out = nullptr;
    verkv_ctx* h = new (std::nothrow) verkv_ctx();
    if (!h) return VERKV_ENOMEM;
    Ctx& ctx = h->c;
    ctx.cfg = *cfg;
    verkv_status st = VERKV_OK;
    const verkv_config& c = ctx.cfg;
    if (c.n_layers <= 0 || c.n_seqs <= 0 || c.max_batch <= 0 || c.n_kv_heads <= 0 || c.n_q_heads <= 0 ||
        c.max_tokens <= 0 || c.n_sink < 0 || c.n_local < 0 || c.n_q_heads % c.n_kv_heads != 0 ||
        !(c.eta > 0.0 && c.eta <= 1.0) || (c.kv_dtype != VERKV_DTYPE_BF16 && c.kv_dtype != VERKV_DTYPE_F32) ||
        (c.sketch != VERKV_SKETCH_EXACT && c.sketch != VERKV_SKETCH_INT8 && c.sketch != VERKV_SKETCH_2BIT) ||
        (c.shrinkage != VERKV_SHRINK_CLIPPED && c.shrinkage != VERKV_SHRINK_BINARY))
        st = fail(ctx, VERKV_EINVAL, "invalid configuration");
    else if (c.head_dim != kHeadDim)
        st = fail(ctx, VERKV_EUNSUPPORTED, "only head_dim 128 is built");
    else if (c.max_batch > decode_max_batch())
        st = fail(ctx, VERKV_EUNSUPPORTED, "max_batch above the built maximum (32)");
    else if (c.sketch == VERKV_SKETCH_2BIT && c.sketch_group != 128)
        st = fail(ctx, VERKV_EUNSUPPORTED, "the 2-bit sketch is built for groups of 128 tokens");
    else if ((long long)c.max_tokens > (1ll << 26))
        st = fail(ctx, VERKV_EUNSUPPORTED, "max_tokens above 2^26");
    if (st == VERKV_OK) {
        ctx.G = c.n_q_heads / c.n_kv_heads;
        if (ctx.G != 1 && ctx.G != 2 && ctx.G != 4 && ctx.G != 8)
            st = fail(ctx, VERKV_EUNSUPPORTED, "GQA group must be 1, 2, 4 or 8");
    }
    if (st == VERKV_OK) {
        ctx.elt = c.kv_dtype == VERKV_DTYPE_BF16 ? 2 : 4;
        cudaGetDevice(&ctx.device);
        int nsm = 0;
        if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, ctx.device) == cudaSuccess && nsm > 0)
            ctx.num_sms = nsm;
        ctx.slots.resize((size_t)c.n_layers * c.n_seqs);
        st = alloc_ws(ctx);
    }
    if (st != VERKV_OK) {
        free_ws(ctx);
        delete h;
        return st;
    }
    *out = h;
    return VERKV_OK;
}

verkv_status verkv_destroy(verkv_ctx* h)
{
    if (!h) return VERKV_EINVAL;
    for (cudaEvent_t e : h->c.ev) cudaEventDestroy(e);
    for (Slot& s : h->c.slots) free_slot(s);
    free_ws(h->c);
    delete h;
    return VERKV_OK;
}

verkv_status verkv_compress(verkv_ctx* h, int32_t layer, int32_t seq, int32_t n_tokens, const void* kv_host,
                            const void* kv_dev, const float* obs_q, int32_t W, const float* tau, verkv_stream stream,
                            verkv_head_stats* stats)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    const verkv_config& c = ctx.cfg;
    if (!slot_ok(ctx, layer, seq)) return fail(ctx, VERKV_EINVAL, "layer/seq slot out of range");
    if (n_tokens <= 0 || n_tokens > c.max_tokens || n_tokens < c.n_sink + c.n_local)
        return fail(ctx, VERKV_EINVAL, "n_tokens out of range");
    if (!(c.eta * (double)n_tokens > (double)(c.n_sink + c.n_local)))
        return fail(ctx, VERKV_EINVAL, "eta * n does not cover the sink and local tokens");
    if (!kv_host) return fail(ctx, VERKV_EINVAL, "kv_host is required (the offloaded cache)");
    if (!obs_q && !tau) return fail(ctx, VERKV_EINVAL, "either obs_q or tau is required");
    if (obs_q && W <= 0) return fail(ctx, VERKV_EINVAL, "W must be positive");
    if ((reinterpret_cast<uintptr_t>(kv_host) & 15) || (reinterpret_cast<uintptr_t>(kv_dev) & 15))
        return fail(ctx, VERKV_EINVAL, "K/V buffers must be 16-byte aligned");
    ctx.last_launches = 0;
    Slot& s = ctx.slot(layer, seq);
    verkv_status rc = compress_slot(ctx, s, layer, seq, n_tokens, kv_host, kv_dev, obs_q, W, tau, (cudaStream_t)stream);
    if (rc != VERKV_OK) {
        cudaStreamSynchronize((cudaStream_t)stream);
        free_slot(s);
        return rc;
    }
    if (stats) std::copy(s.stats.begin(), s.stats.end(), stats);
    return VERKV_OK;
}

verkv_status verkv_decode(verkv_ctx* h, int32_t layer, const int32_t* seq_ids, int32_t B, const float* q, double eps,
                          double delta, float* out, verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    const verkv_config& c = ctx.cfg;
    if (layer < 0 || layer >= c.n_layers) return fail(ctx, VERKV_EINVAL, "layer out of range");
    if (!seq_ids || B <= 0 || B > c.max_batch) return fail(ctx, VERKV_EINVAL, "bad batch");
    if (!q || !out) return fail(ctx, VERKV_EINVAL, "q and out are required");
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 3))
        return fail(ctx, VERKV_EINVAL, "q must be 16-byte aligned");
    if (!(eps >= 0.0) || !std::isfinite(eps)) return fail(ctx, VERKV_EINVAL, "eps must be finite and >= 0");
    if (!(delta > 0.0 && delta < 1.0)) return fail(ctx, VERKV_EINVAL, "delta must lie in (0, 1)");
    if (take_device_timeout(ctx)) return fail(ctx, VERKV_ETIMEOUT, "a bounded device-side wait gave up in an earlier call");
    for (int b = 0; b < B; ++b) {
        if (seq_ids[b] < 0 || seq_ids[b] >= c.n_seqs) return fail(ctx, VERKV_EINVAL, "seq id out of range");
        if (!ctx.slot(layer, seq_ids[b]).live) return fail(ctx, VERKV_ESTATE, "slot was not compressed");
        for (int b2 = 0; b2 < b; ++b2)
            if (seq_ids[b2] == seq_ids[b]) return fail(ctx, VERKV_EINVAL, "duplicate seq id in a batch");
    }
    return decode_rows(ctx, layer, seq_ids, B, q, eps, delta, out, (cudaStream_t)stream);
}

verkv_status verkv_release(verkv_ctx* h, int32_t layer, int32_t seq)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (!slot_ok(ctx, layer, seq)) return fail(ctx, VERKV_EINVAL, "layer/seq slot out of range");
    VK_CUDA(cudaDeviceSynchronize());
    free_slot(ctx.slot(layer, seq));
    return VERKV_OK;
}

verkv_status verkv_get_compress_state(verkv_ctx* h, int32_t layer, int32_t seq, int32_t kv_head, double* cval,
                                      float* tau, float* r, uint8_t* flags, verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (!slot_ok(ctx, layer, seq) || kv_head < 0 || kv_head >= ctx.cfg.n_kv_heads)
        return fail(ctx, VERKV_EINVAL, "slot or head out of range");
    Slot& s = ctx.slot(layer, seq);
    if (!s.live) return fail(ctx, VERKV_ESTATE, "slot was not compressed");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t off = (size_t)kv_head * s.n;
    if (tau) VK_CUDA(cudaMemcpyAsync(tau, s.tau + off, sizeof(float) * s.n, cudaMemcpyDeviceToHost, st));
    if (r) VK_CUDA(cudaMemcpyAsync(r, s.r + off, sizeof(float) * s.n, cudaMemcpyDeviceToHost, st));
    if (flags) VK_CUDA(cudaMemcpyAsync(flags, s.flags + off, s.n, cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    if (cval) *cval = s.stats[kv_head].c;
    return VERKV_OK;
}

verkv_status verkv_get_sketch(verkv_ctx* h, int32_t layer, int32_t seq, int32_t kv_head, int8_t* codes_i8,
                              float* scale_f32, int32_t* pairs, uint8_t* codes_2bit, uint16_t* zero_f16,
                              uint16_t* scale_f16, verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (!slot_ok(ctx, layer, seq) || kv_head < 0 || kv_head >= ctx.cfg.n_kv_heads)
        return fail(ctx, VERKV_EINVAL, "slot or head out of range");
    Slot& s = ctx.slot(layer, seq);
    if (!s.live) return fail(ctx, VERKV_ESTATE, "slot was not compressed");
    cudaStream_t st = (cudaStream_t)stream;
    const size_t n = s.n, off = (size_t)kv_head * n;
    if (ctx.cfg.sketch == VERKV_SKETCH_INT8) {
        if (codes_i8) VK_CUDA(cudaMemcpyAsync(codes_i8, s.codes8 + off * kHeadDim, n * kHeadDim, cudaMemcpyDeviceToHost, st));
        if (scale_f32) VK_CUDA(cudaMemcpyAsync(scale_f32, s.scale8 + off, sizeof(float) * n, cudaMemcpyDeviceToHost, st));
        VK_CUDA(cudaStreamSynchronize(st));
        return VERKV_OK;
    }
    if (ctx.cfg.sketch == VERKV_SKETCH_2BIT) {
        const size_t ng = (n + ctx.cfg.sketch_group - 1) / ctx.cfg.sketch_group, kept = kHeadDim / 4;
        std::vector<uint64_t> packed(n);
        VK_CUDA(cudaMemcpyAsync(packed.data(), s.codes2 + off, sizeof(uint64_t) * n, cudaMemcpyDeviceToHost, st));
        if (pairs) VK_CUDA(cudaMemcpyAsync(pairs, s.pairs + (size_t)kv_head * (kHeadDim / 8), sizeof(int32_t) * (kHeadDim / 8),
                                           cudaMemcpyDeviceToHost, st));
        if (zero_f16) VK_CUDA(cudaMemcpyAsync(zero_f16, s.zero2 + (size_t)kv_head * ng * kept, 2 * ng * kept,
                                              cudaMemcpyDeviceToHost, st));
        if (scale_f16) VK_CUDA(cudaMemcpyAsync(scale_f16, s.scale2 + (size_t)kv_head * ng * kept, 2 * ng * kept,
                                               cudaMemcpyDeviceToHost, st));
        VK_CUDA(cudaStreamSynchronize(st));
        if (codes_2bit)
            for (size_t i = 0; i < n; ++i)
                for (size_t j = 0; j < kept; ++j) codes_2bit[i * kept + j] = (uint8_t)((packed[i] >> (2 * j)) & 3u);
        return VERKV_OK;
    }
    return fail(ctx, VERKV_EINVAL, "the exact sketch has no codes");
}

verkv_status verkv_get_decode_trace(verkv_ctx* h, verkv_row_trace* out, int32_t n_rows, verkv_stream stream)
{
    if (!h || !out) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    const int rows = ctx.last_B * ctx.cfg.n_q_heads;
    if (n_rows < rows) return fail(ctx, VERKV_EINVAL, "n_rows smaller than B * n_q_heads of the last decode");
    std::vector<RowState> rs(rows);
    VK_CUDA(cudaMemcpyAsync(rs.data(), ctx.rows, sizeof(RowState) * rows, cudaMemcpyDeviceToHost, (cudaStream_t)stream));
    VK_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
    if (take_device_timeout(ctx)) return fail(ctx, VERKV_ETIMEOUT, "a bounded device-side wait gave up");
    for (int i = 0; i < rows; ++i) {
        verkv_row_trace& t = out[i];
        const RowState& s = rs[i];
        memset(&t, 0, sizeof(t));
        float mf = -INFINITY;
        if ((unsigned)(s.m_tag >> 32) == (unsigned)ctx.gen) {
            const int mi = (int)((unsigned)s.m_tag ^ 0x80000000u);
            const int bits = mi >= 0 ? mi : mi ^ 0x7fffffff;
            memcpy(&mf, &bits, 4);
        }
        t.m = mf;
        t.D = s.D;
        t.beta = s.beta;
        t.sum_a = s.sum_a;
        t.V = s.V;
        t.b = s.b1;
        t.eps_hat = s.eps_hat;
        t.n_l = s.n_l;
        t.kstar = s.kstar;
        t.no_fetch = s.no_fetch;
        t.fallback = s.fallback;
        t.n_fetch = s.n_fetch;
        t.beta_iters = s.beta_iters;
        t.sel_passes = s.sel_passes;
        for (int k = 0; k < 6; ++k) t.phase_ns[k] = s.phase_ns[k];
        t.n_shrunk = s.n_shrunk;
    }
    return VERKV_OK;
}

verkv_status verkv_get_exact_set(verkv_ctx* h, int32_t b, int32_t hq, int32_t* tokens, int32_t cap, int32_t* count,
                                 verkv_stream stream)
{
    if (!h || !count) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (b < 0 || b >= ctx.last_B || hq < 0 || hq >= ctx.cfg.n_q_heads) return fail(ctx, VERKV_EINVAL, "row out of range");
    cudaStream_t st = (cudaStream_t)stream;
    const int row = b * ctx.cfg.n_q_heads + hq;
    RowState rs;
    VK_CUDA(cudaMemcpyAsync(&rs, ctx.rows + row, sizeof(RowState), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    const int k = std::max(0, rs.kstar);
    *count = k;
    const int m = std::min(k, cap);
    if (tokens && m > 0) {
        std::vector<int32_t> all(k);
        VK_CUDA(cudaMemcpyAsync(all.data(), ctx.elist + (size_t)row * ctx.ws_n, sizeof(int32_t) * k,
                                cudaMemcpyDeviceToHost, st));
        VK_CUDA(cudaStreamSynchronize(st));
        std::sort(all.begin(), all.end());
        std::copy(all.begin(), all.begin() + m, tokens);
    }
    return VERKV_OK;
}

verkv_status verkv_get_fetch_set(verkv_ctx* h, int32_t b, int32_t kv, int32_t* tokens, int32_t cap, int32_t* count,
                                 verkv_stream stream)
{
    if (!h || !count) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (b < 0 || b >= ctx.last_B || kv < 0 || kv >= ctx.cfg.n_kv_heads) return fail(ctx, VERKV_EINVAL, "row out of range");
    cudaStream_t st = (cudaStream_t)stream;
    const int idx = b * ctx.cfg.n_kv_heads + kv;
    int cnt = 0;
    VK_CUDA(cudaMemcpyAsync(&cnt, ctx.ucount + idx, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    *count = cnt;
    const int m = std::min(cnt, cap);
    if (tokens && m > 0) {
        VK_CUDA(cudaMemcpyAsync(tokens, ctx.ulist + (size_t)idx * ctx.ws_n, sizeof(int32_t) * m, cudaMemcpyDeviceToHost, st));
        VK_CUDA(cudaStreamSynchronize(st));
    }
    return VERKV_OK;
}

verkv_status verkv_get_fetch_stats(verkv_ctx* h, int32_t b, int32_t kv, int32_t* n_union, int32_t* n_host,
                                   verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (b < 0 || b >= ctx.last_B || kv < 0 || kv >= ctx.cfg.n_kv_heads) return fail(ctx, VERKV_EINVAL, "row out of range");
    cudaStream_t st = (cudaStream_t)stream;
    const int idx = b * ctx.cfg.n_kv_heads + kv;
    int32_t v[2] = {0, 0};
    VK_CUDA(cudaMemcpyAsync(&v[0], ctx.ucount + idx, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaMemcpyAsync(&v[1], ctx.hrows + idx, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    if (n_union) *n_union = v[0];
    if (n_host) *n_host = v[1];
    return VERKV_OK;
}

verkv_status verkv_get_prefetch_stats(verkv_ctx* h, int32_t b, int32_t kv, int32_t* n_copied, int32_t* n_used,
                                      verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (b < 0 || b >= ctx.last_B || kv < 0 || kv >= ctx.cfg.n_kv_heads) return fail(ctx, VERKV_EINVAL, "row out of range");
    cudaStream_t st = (cudaStream_t)stream;
    const int idx = b * ctx.cfg.n_kv_heads + kv;
    int32_t v[2] = {0, 0};
    VK_CUDA(cudaMemcpyAsync(&v[0], ctx.pf_cnt + idx, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaMemcpyAsync(&v[1], ctx.pf_used + idx, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    if (n_copied) *n_copied = ctx.last_pf_cap > 0 ? std::min(v[0], ctx.last_pf_cap) : 0;
    if (n_used) *n_used = v[1];
    return VERKV_OK;
}

verkv_status verkv_set_prefetch(verkv_ctx* h, int32_t rows_per_kv_head)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (rows_per_kv_head < 0 || rows_per_kv_head > 65536)
        return fail(ctx, VERKV_EINVAL, "prefetch rows per KV head must be in [0, 65536]");
    ctx.prefetch_rows = rows_per_kv_head;
    return VERKV_OK;
}

verkv_status verkv_set_timeline(verkv_ctx* h, int32_t on)
{
    if (!h) return VERKV_EINVAL;
    h->c.timeline = on ? 1 : 0;
    return VERKV_OK;
}

verkv_status verkv_get_timeline(verkv_ctx* h, double* out_us, verkv_stream stream)
{
    if (!h || !out_us) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    for (int k = 0; k < VERKV_TIMELINE_N; ++k) out_us[k] = NAN;
    if (!ctx.last_tline || !ctx.tline) return fail(ctx, VERKV_EINVAL, "the last decode recorded no timeline");
    cudaStream_t st = (cudaStream_t)stream;
    unsigned long long t[16];
    VK_CUDA(cudaMemcpyAsync(t, ctx.tline, sizeof(t), cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    const unsigned long long t0 = t[0];
    if (t0 == ~0ull) return fail(ctx, VERKV_EINVAL, "the last decode recorded no timeline");
    // starts (min slots 1..3, unset = ~0) and ends (max slots 8..11, unset = 0), in microseconds after
    // the scoring kernel's first CTA started
    const int slot[VERKV_TIMELINE_N] = {1, 8, 2, 9, 10, 3, 11};
    for (int k = 0; k < VERKV_TIMELINE_N; ++k) {
        const unsigned long long v = t[slot[k]];
        const bool unset = slot[k] < 8 ? v == ~0ull : v == 0ull;
        out_us[k] = unset ? NAN : (double)(long long)(v - t0) * 1e-3;
    }
    return VERKV_OK;
}

verkv_status verkv_set_shortlist(verkv_ctx* h, int32_t k)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (k < 0 || k > kMaxShortlist) return fail(ctx, VERKV_EINVAL, "shortlist size must be in [0, 1024]");
    ctx.shortlist_k = k;
    return VERKV_OK;
}

verkv_status verkv_get_shortlist(verkv_ctx* h, int32_t b, int32_t kv, int32_t* tokens, int32_t cap, int32_t* count,
                                 verkv_stream stream)
{
    if (!h || !count) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (b < 0 || b >= ctx.last_B || kv < 0 || kv >= ctx.cfg.n_kv_heads) return fail(ctx, VERKV_EINVAL, "row out of range");
    cudaStream_t st = (cudaStream_t)stream;
    const int idx = b * ctx.cfg.n_kv_heads + kv;
    int cnt = 0;
    if (ctx.shortlist_k > 0) {
        VK_CUDA(cudaMemcpyAsync(&cnt, ctx.scount + idx, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
        VK_CUDA(cudaStreamSynchronize(st));
    }
    *count = cnt;
    const int m = std::min(cnt, cap);
    if (tokens && m > 0) {
        std::vector<int32_t> li(m);
        VK_CUDA(cudaMemcpyAsync(li.data(), ctx.slist + (size_t)idx * kMaxShortlist, sizeof(int32_t) * m,
                                cudaMemcpyDeviceToHost, st));
        Slot& s = ctx.slot(ctx.last_layer, ctx.last_seq[b]);
        std::vector<int32_t> ltok((size_t)s.stats[kv].n_l);
        if (!ltok.empty())
            VK_CUDA(cudaMemcpyAsync(ltok.data(), s.ltok + (size_t)kv * s.n, sizeof(int32_t) * ltok.size(),
                                    cudaMemcpyDeviceToHost, st));
        VK_CUDA(cudaStreamSynchronize(st));
        for (int i = 0; i < m; ++i) tokens[i] = ltok[li[i]];
        std::sort(tokens, tokens + m);
    }
    return VERKV_OK;
}

verkv_status verkv_set_stage_capacity(verkv_ctx* h, int64_t rows_per_kv_head)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (rows_per_kv_head < VERKV_STAGE_ETA_N)
        return fail(ctx, VERKV_EINVAL, "staging capacity must be VERKV_STAGE_ETA_N, VERKV_STAGE_ALL, 0 or positive");
    ctx.stage_rows = rows_per_kv_head;
    return VERKV_OK;
}

verkv_status verkv_selftest_wait_timeout(verkv_ctx* h, verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    cudaStream_t st = (cudaStream_t)stream;
    VK_CUDA(cudaStreamSynchronize(st));
    if (take_device_timeout(ctx)) return fail(ctx, VERKV_ETIMEOUT, "a bounded device-side wait gave up in an earlier call");
    wait_timeout_kernel<<<1, 32, 0, st>>>(ctx.d_err);
    VK_CUDA(cudaGetLastError());
    VK_CUDA(cudaStreamSynchronize(st));
    if (take_device_timeout(ctx)) return fail(ctx, VERKV_ETIMEOUT, "the self-test wait gave up, as intended");
    return VERKV_OK;
}

verkv_status verkv_set_append_capacity(verkv_ctx* h, int32_t rows_per_kv_head)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (rows_per_kv_head < 0) return fail(ctx, VERKV_EINVAL, "append capacity must be >= 0");
    ctx.append_rows = rows_per_kv_head;
    return VERKV_OK;
}

verkv_status verkv_append(verkv_ctx* h, int32_t layer, int32_t seq, int32_t n_new, const void* kv_new,
                          verkv_stream stream)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (!slot_ok(ctx, layer, seq)) return fail(ctx, VERKV_EINVAL, "layer/seq slot out of range");
    if (n_new < 0 || (n_new > 0 && !kv_new)) return fail(ctx, VERKV_EINVAL, "bad appended rows");
    Slot& s = ctx.slot(layer, seq);
    if (!s.live) return fail(ctx, VERKV_ESTATE, "slot was not compressed");
    if (n_new == 0) return VERKV_OK;
    if ((int64_t)s.n_tail + n_new > s.cap_tail)
        return fail(ctx, VERKV_EINVAL, "appended tokens exceed the room reserved at compress");
    if (reinterpret_cast<uintptr_t>(kv_new) % 16 != 0) return fail(ctx, VERKV_EINVAL, "appended rows must be 16-byte aligned");
    cudaPointerAttributes pa;
    VK_CUDA(cudaPointerGetAttributes(&pa, kv_new));
    if (pa.type == cudaMemoryTypeUnregistered)   // read by a kernel: device or page-locked host memory only
        return fail(ctx, VERKV_EINVAL, "appended rows must be in device or pinned host memory");
    return append_rows(ctx, s, n_new, kv_new, (cudaStream_t)stream);
}

verkv_status verkv_get_appended(verkv_ctx* h, int32_t layer, int32_t seq, int32_t* n_appended)
{
    if (!h || !n_appended) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (!slot_ok(ctx, layer, seq)) return fail(ctx, VERKV_EINVAL, "layer/seq slot out of range");
    Slot& s = ctx.slot(layer, seq);
    if (!s.live) return fail(ctx, VERKV_ESTATE, "slot was not compressed");
    *n_appended = s.n_tail;
    return VERKV_OK;
}

verkv_status verkv_get_row_weights(verkv_ctx* h, int32_t b, int32_t hq, float* w_hat, int32_t* tokens, int32_t cap,
                                   int32_t* count, verkv_stream stream)
{
    if (!h || !count) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (b < 0 || b >= ctx.last_B || hq < 0 || hq >= ctx.cfg.n_q_heads) return fail(ctx, VERKV_EINVAL, "row out of range");
    cudaStream_t st = (cudaStream_t)stream;
    const int row = b * ctx.cfg.n_q_heads + hq;
    const int kv = hq / ctx.G;
    Slot& s = ctx.slot(ctx.last_layer, ctx.last_seq[b]);
    const int nl = s.stats[kv].n_l;
    *count = nl;
    const int m = std::min(nl, cap);
    if (w_hat && m > 0)
        VK_CUDA(cudaMemcpyAsync(w_hat, ctx.wl + (size_t)row * ctx.ws_n, sizeof(float) * m, cudaMemcpyDeviceToHost, st));
    if (tokens && m > 0)
        VK_CUDA(cudaMemcpyAsync(tokens, s.ltok + (size_t)kv * s.n, sizeof(int32_t) * m, cudaMemcpyDeviceToHost, st));
    VK_CUDA(cudaStreamSynchronize(st));
    return VERKV_OK;
}

verkv_status verkv_set_kernel_timing(verkv_ctx* h, int32_t enable)
{
    if (!h) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    if (enable && ctx.ev.empty()) {
        ctx.ev.resize(Ctx::kMaxTimed + 1);
        for (cudaEvent_t& e : ctx.ev) VK_CUDA(cudaEventCreate(&e));
    }
    ctx.timing = enable != 0;
    ctx.n_ev = 0;
    ctx.ev_prev = -1;
    ctx.ev_name.clear();
    ctx.ev_from.clear();
    return VERKV_OK;
}

verkv_status verkv_get_kernel_times(verkv_ctx* h, const char** names, float* ms, int32_t cap, int32_t* count,
                                    verkv_stream stream)
{
    if (!h || !count) return VERKV_EINVAL;
    Ctx& ctx = h->c;
    const int n = (int)ctx.ev_name.size();
    *count = n;
    (void)stream;
    if (n > 0) VK_CUDA(cudaEventSynchronize(ctx.ev[ctx.n_ev - 1]));
    for (int i = 0; i < n && i < cap; ++i) {
        if (names) names[i] = ctx.ev_name[i];
        // entry i ends at the event recorded right after its launch: the i-th non-begin event
        if (ms) VK_CUDA(cudaEventElapsedTime(&ms[i], ctx.ev[ctx.ev_from[i]], ctx.ev[ctx.ev_from[i] + 1]));
    }
    ctx.n_ev = 0;
    ctx.ev_prev = -1;
    ctx.ev_name.clear();
    ctx.ev_from.clear();
    return VERKV_OK;
}

}  // extern "C"
