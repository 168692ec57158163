// Internal state of a libverkv context (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/verkv.h"

namespace verkv {

// Compressed state of one (layer, sequence) slot.  Per-KV-head arrays are laid out
// [n_kv_heads][n] with head stride n (the slot's context length).
struct Slot {
    bool live = false;
    int n = 0;
    int cap_n = 0;              // token capacity of the per-token arrays (reused while n <= cap_n)
    size_t cap_res = 0;         // resident rows kvres can hold
    int n_tail = 0;             // tokens appended since compress (ids n ..): H, rows after each head's H u S
    int cap_tail = 0;           // room for appended rows per KV head, reserved in kvres
    const void* kv_host = nullptr;  // borrowed pinned [Hkv][n][2][d]

    float* tau = nullptr;       // [Hkv][n] importance scores after clamping / forcing
    float* r = nullptr;         // [Hkv][n] inclusion probabilities (fp32)
    uint8_t* flags = nullptr;   // [Hkv][n] 2 = H, 1 = S, 0 = L \ S
    int32_t* lpos = nullptr;    // [Hkv][n] token -> index in L (ascending tokens); -(H index)-1 for H
    int32_t* ltok = nullptr;    // [Hkv][n] L index -> token
    float* rl = nullptr;        // [Hkv][n] r by L index
    int32_t* lslot = nullptr;   // [Hkv][n] L index -> resident slot when the token is in S, else -1
    float2* lq = nullptr;       // [Hkv][n] by L index: ((1 - r) / r, r / (1 - r))
    int32_t* rtok = nullptr;    // [Hkv][n] resident slot -> token (H u S ascending)
    int32_t* hslot = nullptr;   // [Hkv][n] H index -> resident slot
    int32_t* counts = nullptr;  // [Hkv][4] |H|, |L|, |S|, |H|+|S|
    double* c = nullptr;        // [Hkv] water-filling constant
    int32_t* capped = nullptr;  // [Hkv] tokens outside sink/local with r = 1
    void* kvres = nullptr;      // [sum_h (m_h + cap_tail)][2][d] resident K/V rows, head h from res_off[h]:
                                // its m_h rows of H u S, then the appended rows
    int64_t* res_off = nullptr; // device [Hkv + 1] row offsets into kvres

    // sketches
    int8_t* codes8 = nullptr;   // [Hkv][n][d]
    float* scale8 = nullptr;    // [Hkv][n]
    uint64_t* codes2 = nullptr; // [Hkv][n] 2-bit codes of the kept channels, channel j at bits 2j..2j+1
    __half* zero2 = nullptr;    // [Hkv][ngroups][d/4]
    __half* scale2 = nullptr;   // [Hkv][ngroups][d/4]
    int32_t* pairs = nullptr;   // [Hkv][d/8] kept rotate-half pairs, ascending
    double* energy = nullptr;   // [Hkv][d/2] pair energies (scratch of the 2-bit sketch)
    void* kexact = nullptr;     // [Hkv][n][d] keys for the exact sketch

    // rows of L \ S fetched by earlier decodes, kept in device memory (the staging cache)
    int32_t* stage_of = nullptr;   // [Hkv][n] token -> staged row of its head (-1: not staged)
    void* stage = nullptr;         // [sum_h cap_h][2][d] staged K/V rows, head h from stage_off[h]
    int64_t* stage_off = nullptr;  // device [Hkv + 1] row offsets into stage (cap_h = difference)
    int32_t* stage_cnt = nullptr;  // [Hkv] rows staged so far
    size_t cap_stage = 0;          // rows stage can hold
    std::vector<int64_t> stage_off_host;

    std::vector<verkv_head_stats> stats;     // host copy
    std::vector<int64_t> res_off_host;       // host copy of res_off
};

// Per query row scalars of one decode (device).  Doubles are accumulated with atomics.
struct RowState {
    unsigned long long m_tag;  // (decode generation << 32) | order-preserving bits of the max logit m
    int m_pad;
    int no_fetch;
    int kstar;
    int fallback;
    int n_l;
    int n_h;
    int n_fetch;        // |E \ S|
    int b_arg;          // L index of the largest b_i
    double D;           // sum_H w + sum_L w^
    double alpha_sum;   // sum_L w^ (1 - r): upper end of the beta bracket
    double beta;
    double sum_a;
    double V;
    double b1, b2;      // largest and second-largest b_i
    double eps_hat;
    float beta_f;       // beta in fp32 (what the attention weights use)
    int n_shrunk;       // binary shrinkage: entries given lambda = r
    int beta_iters;     // passes of the beta solve
    int sel_passes;     // radix-select passes
    unsigned int phase_ns[6];  // decide kernel: ns spent in phases 0..4 and in the ranking (rank 0)
};

constexpr int kMaxShortlist = 1024;    // largest shortlist per KV head
constexpr int kShortlistBins = 4096;   // shortlist radix select: first-level bins (top 12 key bits)

struct Ctx {
    verkv_config cfg{};
    int device = 0;
    int G = 1;                      // query heads per KV head
    size_t elt = 2;                 // bytes per K/V element
    std::vector<Slot> slots;        // [n_layers * n_seqs]
    std::string err;
    int last_launches = 0;

    // optional per-kernel timing: events recorded between launches on the call's stream, kept
    // across calls until read (verkv_get_kernel_times)
    static constexpr int kMaxTimed = 4096;
    bool timing = false;
    std::vector<cudaEvent_t> ev;          // pool of kMaxTimed + 1 events
    std::vector<const char*> ev_name;     // entry i: kernel name
    std::vector<int> ev_from;             // entry i: event index before the kernel
    int n_ev = 0;                         // events used
    int ev_prev = -1;                     // event recorded last
    int gen = 0;                          // decode generation tag

    // decode workspace, sized for max_batch rows sets
    int ws_rows = 0;                // max_batch * n_q_heads
    int ws_n = 0;                   // max_tokens
    int ws_npow2 = 0;               // next power of two >= max_tokens
    float2* tl = nullptr;           // [rows][n] sketch logits (hi, lo) by L index
    float2* th = nullptr;           // [rows][n] exact logits by H index
    float* wl = nullptr;            // [rows][n] sketch weights by L index
    RowState* rows = nullptr;       // [rows]
    unsigned long long* keys = nullptr;  // [rows][npow2] gain keys (full-row path)
    int32_t* mark = nullptr;        // [rows][n] generation tag: L index made exact (full-row path)
    int32_t* elist = nullptr;       // [rows][n] tokens made exact
    uint32_t* ebits = nullptr;      // [rows][n/32 + 1] per query row: tokens of L_g[:k*] \ S (bitmap)
    float* om = nullptr;            // [rows][n] per query row: weight factor of each resident slot
    int32_t* ulist = nullptr;       // [max_batch][Hkv][n] fetched union, ascending tokens
    uint8_t* umask = nullptr;       // [max_batch][Hkv][n] query heads (bit g) whose exact set holds the row
    int32_t* adone = nullptr;       // [max_batch][Hkv] attention blocks finished (zero between calls)
    int32_t* ucount = nullptr;      // [max_batch][Hkv]
    float* part = nullptr;          // [rows][nsplit][d + 2] attention partials
    int nsplit = 128;               // largest split of the attention over blocks per KV head
    int num_sms = 152;              // multiprocessors of the context's device
    int32_t* hrows = nullptr;       // [max_batch][Hkv] rows the last decode read over the host link
    int shortlist_k = 0;            // App. A.1 shortlist per KV head (0: off)
    int32_t* slist = nullptr;       // [max_batch][Hkv][kMaxShortlist] L indices of the last shortlist
    int32_t* scount = nullptr;      // [max_batch][Hkv] its size
    uint32_t* shist = nullptr;      // [max_batch][Hkv][kShortlistBins + 1] shortlist first-level histogram + count
                                    // (zero between calls)
    int64_t stage_rows = VERKV_STAGE_ETA_N;   // staging capacity per KV head and slot (verkv_set_stage_capacity)
    // speculative prefetch (verkv_set_prefetch): while the decision runs, rows of L \ S with the
    // largest alpha = w^ (1 - r) are copied from pinned host memory into a per-call device buffer, and
    // the attention reads the ones it needs from there
    int prefetch_rows = 4096;       // rows per (sequence, KV head) a decode may copy ahead (0: off)
    int pf_cap = 0;                 // rows per (sequence, KV head) the buffers below hold
    unsigned long long* tline = nullptr;   // decode call timeline (16 device times), when enabled
    int timeline = 0;               // verkv_set_timeline
    int last_tline = 0;             // the last decode recorded one
    void* tau_ws = nullptr;         // compress: importance-score scratch (partials, row stats, raw scores)
    size_t tau_ws_cap = 0;
    void* pf_buf = nullptr;         // [max_batch][Hkv][pf_cap][2][d] rows copied ahead
    int32_t* pf_of = nullptr;       // [max_batch][Hkv][max_tokens] token -> prefetch row (valid when pf_tok agrees)
    int32_t* pf_tok = nullptr;      // [max_batch][Hkv][pf_cap] prefetch row -> token, this call
    int32_t* pf_cnt = nullptr;      // [max_batch][Hkv] rows claimed this call (reset by the scoring kernel)
    int32_t* pf_used = nullptr;     // [max_batch][Hkv] prefetched rows the attention read (reset likewise)
    unsigned long long* dprog = nullptr;  // (decode generation << 32) | query rows decided so far
    int last_pf_cap = 0;            // pf_cap of the last decode (0: the prefetch did not run)
    int append_rows = 0;            // room reserved per KV head and slot for decode-time appended tokens
    int* h_err = nullptr;           // mapped pinned host word: a device-side bounded wait gave up
    int* d_err = nullptr;           // its device address

    // per-decode small arrays
    int32_t* d_slot_n = nullptr;    // [max_batch] n of each row set's slot
    int last_B = 0;
    int last_layer = -1;
    std::vector<int> last_seq;
    std::vector<int> last_n;

    Slot& slot(int layer, int seq) { return slots[(size_t)layer * cfg.n_seqs + seq]; }
};

// Slot pointers for the decode kernels (device-side copy, one entry per b).
struct SlotView {
    int n;
    int n_tail;                  // appended tokens (H), rows m_h .. m_h + n_tail - 1 of the head in kvres
    const float* r;
    const uint8_t* flags;
    const int32_t* lpos;
    const int32_t* ltok;
    const float* rl;
    const int32_t* lslot;
    const float2* lq;
    const int32_t* rtok;
    const int32_t* hslot;
    const int32_t* counts;
    const void* kvres;
    const int64_t* res_off;
    const void* kv_host;
    const int8_t* codes8;
    const float* scale8;
    const uint64_t* codes2;
    const __half* zero2;
    const __half* scale2;
    const int32_t* pairs;
    const void* kexact;
    int32_t* stage_of;           // nullptr: staging off for this slot
    void* stage;
    const int64_t* stage_off;
    int32_t* stage_cnt;
};

verkv_status compress_slot(Ctx& ctx, Slot& s, int layer, int seq, int n, const void* kv_host, const void* kv_dev,
                           const float* obs_q, int W, const float* tau, cudaStream_t st);
verkv_status decode_rows(Ctx& ctx, int layer, const int32_t* seq_ids, int B, const float* q, double eps,
                         double delta, float* out, cudaStream_t st);
void free_slot(Slot& s);
verkv_status append_rows(Ctx& ctx, Slot& s, int n_new, const void* src, cudaStream_t st);

}  // namespace verkv

#define VK_CUDA(call)                                                                        \
    do {                                                                                     \
        cudaError_t e_ = (call);                                                             \
        if (e_ != cudaSuccess) {                                                             \
            ctx.err = std::string(#call) + ": " + cudaGetErrorString(e_);                    \
            return e_ == cudaErrorMemoryAllocation ? VERKV_ENOMEM : VERKV_ECUDA;            \
        }                                                                                    \
    } while (0)

// After every kernel launch: check the launch, count it, and (when timing) record an event.
#define VK_LAUNCHED(name)                                                                    \
    do {                                                                                     \
        cudaError_t e_ = cudaGetLastError();                                                 \
        if (e_ != cudaSuccess) {                                                             \
            ctx.err = std::string("kernel launch (") + (name) + "): " + cudaGetErrorString(e_); \
            return VERKV_ECUDA;                                                              \
        }                                                                                    \
        ++ctx.last_launches;                                                                 \
        if (ctx.timing && ctx.ev_prev >= 0 && ctx.n_ev < verkv::Ctx::kMaxTimed) {            \
            ctx.ev_name.push_back(name);                                                     \
            ctx.ev_from.push_back(ctx.ev_prev);                                              \
            cudaEventRecord(ctx.ev[ctx.n_ev], st);                                           \
            ctx.ev_prev = ctx.n_ev++;                                                        \
        }                                                                                    \
    } while (0)

// Start of a timed call.
#define VK_TIMING_BEGIN()                                                                    \
    do {                                                                                     \
        ctx.ev_prev = -1;                                                                    \
        if (ctx.timing && ctx.n_ev < verkv::Ctx::kMaxTimed) {                                \
            cudaEventRecord(ctx.ev[ctx.n_ev], st);                                           \
            ctx.ev_prev = ctx.n_ev++;                                                        \
        }                                                                                    \
    } while (0)
