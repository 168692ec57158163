"""Shared drivers for the parity tests: run one workload through the CUDA library (via the C ABI)
and through the oracle, from the same seeded inputs.  Nothing computed by the CUDA path is ever fed
to the oracle."""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

import oracle
from verified_kv_cache_gb300 import workloads

G_GAP = 1e-6      # fetched-set exemption: oracle gains closer than this (relative) at the k* boundary
K_GAP = 1e-6      # k* exemption: residual certificate within this (relative) of eps
B_GAP = 1e-6      # binary shrinkage: the oracle's stop test gamma > 2 beta within this (relative) of equality
REL_SCALAR = 1e-4 # c, beta, eps_hat
REL_OUT = 2e-3    # attention output, relative L2
# fp32 weights w^ = exp(t - m) underflow below 2^-126 of the row maximum; scale-free scalars (eps_hat,
# beta / D) smaller than this floor are zero on the device.
ABS_FLOOR = 1e-30


# ----------------------------------------------------------------------------- oracle side
@dataclass
class OracleSlot:
    tau: np.ndarray          # [Hkv, n] fp32
    c: np.ndarray            # [Hkv]
    r32: np.ndarray          # [Hkv, n]
    r64: np.ndarray
    flags: np.ndarray        # [Hkv, n]
    sketch: dict = field(default_factory=dict)


def oracle_tau(w: workloads.Workload, b: int) -> np.ndarray:
    G, W = w.group, w.obs_q.shape[2]
    out = np.zeros((w.n_kv, w.n), np.float32)
    for h in range(w.n_kv):
        Q = w.obs_q[b, h * G:(h + 1) * G].reshape(G * W, w.d)
        out[h] = oracle.tau(w.K[b, h], Q, w.n_sink, w.n_local)
    return out


def oracle_compress(w: workloads.Workload, b: int, tau: np.ndarray, layer: int = 0, seq: int = 0,
                    seed: int | None = None) -> OracleSlot:
    seed = w.seed if seed is None else seed
    Hkv, n = w.n_kv, w.n
    c = np.zeros(Hkv)
    r32 = np.zeros((Hkv, n), np.float32)
    r64 = np.zeros((Hkv, n))
    flags = np.zeros((Hkv, n), np.uint8)
    sk = {}
    for h in range(Hkv):
        c[h], _, r64[h], r32[h] = oracle.waterfill(tau[h], w.n_sink, w.n_local, w.eta * n)
        flags[h] = oracle.poisson_sample(r32[h], seed, h, layer, seq)
        if w.sketch == "int8":
            sk[h] = oracle.sketch_int8(w.K[b, h])
        elif w.sketch == "2bit":
            sk[h] = oracle.sketch_2bit(w.K[b, h])
    return OracleSlot(tau, c, r32, r64, flags, sk)


def oracle_sketch_logits(w, b, h, q, slot: OracleSlot):
    if w.sketch == "exact":
        return oracle.logits_exact(q, w.K[b, h])
    if w.sketch == "int8":
        codes, scale = slot.sketch[h]
        return oracle.logits_int8(q, codes, scale)
    pairs, codes, zero, scale = slot.sketch[h]
    return oracle.logits_2bit(q, pairs, codes, zero, scale)


def oracle_decode(w, b, slot: OracleSlot, q_bh: np.ndarray, eps, delta, mode=1, shrinkage=0, shortlist=0):
    """q_bh: [Hq, d] for sequence b.  Returns per row dicts and per KV head fetch unions and outputs.
    shrinkage: 0 = clipped coefficients (Definition 2), 1 = binary (Appendix A.2).
    shortlist: k > 0 uses exact weights for the sampled tokens and the Appendix A.1 shortlist of k
    tokens per KV head (each row dict then carries the head's shortlist mask and scores).
    When w holds more tokens than the slot (w.n > len(slot.flags[h])), the extra tokens are ones
    appended at decode time: they join H (r = 1) and have no sketch."""
    G = w.group
    n0 = slot.flags.shape[1]
    tail = w.n - n0
    flags = np.concatenate([slot.flags, np.full((w.n_kv, tail), 2, np.uint8)], axis=1)
    r32 = np.concatenate([slot.r32, np.ones((w.n_kv, tail), np.float32)], axis=1)
    rows = []
    logits = {}
    for hq in range(w.n_q):
        q = q_bh[hq].astype(np.float64)
        h = hq // G
        ts = oracle_sketch_logits(w, b, h, q, slot)
        ts = np.concatenate([ts[:n0], np.zeros(tail)])
        logits[hq] = (oracle.logits_exact(q, w.K[b, h]), ts)
    masks = {}
    if shortlist > 0:
        for h in range(w.n_kv):
            ts_rows = np.stack([logits[h * G + g][1] for g in range(G)])
            sl = oracle.shortlist(flags[h], ts_rows, shortlist)
            masks[h] = (sl, ts_rows.max(axis=0))
    for hq in range(w.n_q):
        h = hq // G
        te, ts = logits[hq]
        use = None
        if shortlist > 0:
            use = masks[h][0] | (flags[h] == 1)
        res = oracle.kvfetch_row(flags[h], r32[h], te, ts, eps, delta, mode=mode, shrinkage=shrinkage,
                                 use_exact=use)
        if shortlist > 0:
            res["shortlist"], res["sl_score"] = masks[h]
        if shrinkage == 1:
            Lm = flags[h] != 2
            res["w_l"] = np.exp((ts if use is None else np.where(use, te, ts))[Lm] - res["m"])
            res["r_l"] = r32[h][Lm].astype(np.float64)
            res["n_shrunk"] = int((res["lam"][Lm] < 1.0).sum())
        res["out"] = oracle.attention_row(flags[h], r32[h], te, w.V[b, h], res["lam"], res["exact_mask"])
        # what the output check of an exempted row needs: the row's state, logits and values
        res["_flags"], res["_r32"], res["_te"], res["_ts"], res["_V"] = flags[h], r32[h], te, ts, w.V[b, h]
        rows.append(res)
    unions = []
    for h in range(w.n_kv):
        u = np.zeros(w.n, bool)
        for g in range(G):
            u |= rows[h * G + g]["exact_mask"] & (flags[h] == 0)
        unions.append(np.nonzero(u)[0])
    return rows, unions


# ----------------------------------------------------------------------------- CUDA side
class GpuCase:
    """Holds the device/pinned buffers of one workload for the library."""

    def __init__(self, w: workloads.Workload, lib_ctx, layers=1):
        import torch
        self.w = w
        self.ctx = lib_ctx
        self.kv_host = []
        self.kv_dev = []
        self.obs = []
        for b in range(w.batch):
            arr = w.kv_host_layout(b)
            t = torch.from_numpy(arr)
            if w.kv_dtype == "bf16":
                t = t.view(torch.bfloat16)
            pinned = t.pin_memory()
            self.kv_host.append(pinned)
            self.kv_dev.append(pinned.to("cuda"))
            self.obs.append(torch.from_numpy(np.ascontiguousarray(w.obs_q[b])).to("cuda"))

    def compress(self, b, layer=0, seq=None, tau=None, use_dev=True):
        import torch
        seq = b if seq is None else seq
        tau_t = None
        if tau is not None:
            tau_t = torch.from_numpy(np.ascontiguousarray(tau, np.float32)).to("cuda")
        stats = self.ctx.compress(layer, seq, self.w.n, self.kv_host[b], self.kv_dev[b] if use_dev else None,
                                  None if tau is not None else self.obs[b], self.w.obs_q.shape[2], tau_t)
        torch.cuda.synchronize()
        return stats

    def decode(self, q_step: np.ndarray, eps, delta, layer=0, seq_ids=None):
        import torch
        B = q_step.shape[0]
        seq_ids = list(range(B)) if seq_ids is None else seq_ids
        q = torch.from_numpy(np.ascontiguousarray(q_step, np.float32)).to("cuda")
        out = torch.empty_like(q)
        self.ctx.decode(layer, seq_ids, q, eps, delta, out)
        torch.cuda.synchronize()
        return out.cpu().numpy()


def make_lib_ctx(w, n_layers=1, n_seqs=None, max_batch=None, max_tokens=None, shrinkage="clipped"):
    from verified_kv_cache_gb300 import binding
    return binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=max_tokens or w.n, head_dim=w.d,
                         n_layers=n_layers, n_seqs=n_seqs or w.batch, max_batch=max_batch or w.batch,
                         n_sink=w.n_sink, n_local=w.n_local, eta=w.eta, seed=w.seed, sketch=w.sketch,
                         kv_dtype=w.kv_dtype, shrinkage=shrinkage)


# ----------------------------------------------------------------------------- comparisons
def rel(a, b):
    return abs(a - b) / max(abs(b), 1e-300)


def close(a, b, rtol=REL_SCALAR, atol=ABS_FLOOR):
    return abs(a - b) <= rtol * abs(b) + atol


def _gamma_order(orow):
    w, r = orow["w_l"], orow["r_l"]
    g = w * (1 - r) / r
    return w, r, g, np.lexsort((np.arange(len(g)), -g))


def binary_boundary_is_near_tie(orow, k_a, k_b):
    """Binary shrinkage: the device shrank k_a entries of the gamma order, the oracle k_b.  Exempt
    when the oracle's own test gamma_(k) > 2 beta_k sits within B_GAP (relative) of equality at every
    position between the two."""
    w, r, g, order = _gamma_order(orow)
    pre = np.concatenate([[0.0], np.cumsum((w * (1 - r))[order])])
    for k in range(min(k_a, k_b), max(k_a, k_b) + 1):
        if k >= len(g):
            continue
        gk = g[order[k]]
        if abs(gk - 2 * pre[k]) > B_GAP * gk:
            return False
    return True


def binary_boundary_underflows(orow, k_a, k_b):
    """The entries between the two prefix ends have weights below ABS_FLOOR of D: they are zero in the
    device's fp32 weights (which never shrinks an entry of weight 0) and move no checked quantity."""
    w, r, g, order = _gamma_order(orow)
    between = order[min(k_a, k_b):max(k_a, k_b)]
    return bool(np.all(w[between] <= ABS_FLOOR * orow["D"]))


def check_row(gpu_trace, gpu_set, orow, eps, flags_h):
    """Compare one query row.  Returns 'ok', 'exempt-b', 'exempt-k' or 'exempt-g'; raises on a real
    mismatch."""
    if "n_shrunk" in orow and gpu_trace["n_shrunk"] != orow["n_shrunk"]:
        kg, ko = gpu_trace["n_shrunk"], orow["n_shrunk"]
        if not binary_boundary_underflows(orow, kg, ko):
            assert binary_boundary_is_near_tie(orow, kg, ko), ("binary shrinkage prefix differs", kg, ko)
            return "exempt-b"
    assert close(gpu_trace["eps_hat"], orow["eps_hat"]), (gpu_trace["eps_hat"], orow["eps_hat"])
    assert close(gpu_trace["beta"] / gpu_trace["D"], orow["beta"] / orow["D"]), (gpu_trace, orow["beta"], orow["D"])
    nf_o = bool(orow["no_fetch"])
    if bool(gpu_trace["no_fetch"]) != nf_o:
        assert abs(orow["eps_hat"] - eps) <= K_GAP * eps, ("no-fetch decision differs", gpu_trace, orow["eps_hat"])
        return "exempt-k"
    if nf_o:
        assert gpu_trace["kstar"] == 0 and len(gpu_set) == 0
        return "ok"
    o_set = np.nonzero(orow["exact_mask"])[0]
    k_o, k_g = int(orow["kstar"]), int(gpu_trace["kstar"])
    if k_o != k_g:
        lo, hi = min(k_o, k_g), max(k_o, k_g)
        resid = orow["resid"]
        # every residual certificate between the two answers must sit within K_GAP of eps
        band = resid[lo:hi]
        assert np.all(np.abs(band - eps) <= K_GAP * eps), ("k* differs", k_o, k_g, band, eps)
        return "exempt-k"
    if np.array_equal(np.sort(gpu_set), o_set):
        return "ok"
    diff = np.setxor1d(gpu_set, o_set)
    g = orow["gain"]
    order = orow["order"]
    g_in = g[order[k_o - 1]]
    g_out = g[order[k_o]] if k_o < len(order) else 0.0
    assert g_in - g_out <= G_GAP * g_in, ("fetched set differs beyond the gain-gap exemption", diff[:10], g_in, g_out)
    assert np.all(np.abs(g[diff] - g_in) <= G_GAP * g_in), ("set difference outside the boundary band", diff[:10])
    return "exempt-g"


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def output_with_device_decision(orow, gpu_set, n_shrunk=None):
    """The oracle's output for a row whose decision took an exemption: the oracle's coefficients and
    the DEVICE's exact set (and, for binary shrinkage, the device's shrunk prefix of the oracle's gamma
    order), so that the attention of every row is checked even where the decision legitimately differs."""
    flags, r32, te, V = orow["_flags"], orow["_r32"], orow["_te"], orow["_V"]
    lam = orow["lam"]
    if n_shrunk is not None and "w_l" in orow and n_shrunk != orow["n_shrunk"]:
        _, r, _, order = _gamma_order(orow)
        Lm = flags != 2
        lam_l = np.ones(int(Lm.sum()))
        lam_l[order[:n_shrunk]] = r[order[:n_shrunk]]
        lam = np.zeros(len(flags))
        lam[Lm] = lam_l
    mask = np.zeros(len(flags), bool)
    mask[np.asarray(gpu_set, np.int64)] = True
    return oracle.attention_row(flags, r32, te, V, lam, mask)


def check_row_output(gpu_trace, gpu_set, orow, eps, out_row, ctx_msg=None):
    """check_row, then the attention output of the row within REL_OUT: against the oracle's own output
    when the decision matched, else against the oracle's output over the device's decision."""
    verdict = check_row(gpu_trace, gpu_set, orow, eps, None)
    ref = orow["out"] if verdict == "ok" else output_with_device_decision(orow, gpu_set, gpu_trace.get("n_shrunk"))
    err = rel_l2(np.asarray(out_row, np.float64), ref)
    assert err <= REL_OUT, (ctx_msg, verdict, err)
    return verdict
