"""The allocation-free decision entry point, verkv_certify_row_static.

It exists for callers that cannot call cudaMalloc: engines that fix their device memory up front
(their own arena, a real-time loop that must not allocate) and code running while a CUDA stream is
captured into a graph, where an allocation would fail or become part of the graph.  It takes one query
row's sketch weights and inclusion probabilities and returns beta, eps_hat, k* and the tokens to make
exact, using a static device array as its only scratch.

Checked through the C ABI against the decision verkv_decode makes for the same rows (the existing
entry point) and against the oracle's decision, each on two calls in a row (the static scratch keeps
the previous call's contents).  The file is collected last so that a run stopping at the first
failure has run every other test before it.
"""
import ctypes
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from verified_kv_cache_gb300 import binding, build, workloads

from vkcase import check_row

pytestmark = pytest.mark.gpu


def _static_fn():
    L = binding.lib()
    f = L.verkv_certify_row_static
    P = ctypes.c_void_p
    f.argtypes = [P, P, ctypes.c_int32, ctypes.c_double, ctypes.c_double, ctypes.c_double, P, P, P, P]
    f.restype = ctypes.c_int
    return f


def test_static_certificate_matches_decode_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    f = _static_fn()
    w = workloads.qwen_layer_case(seed=31, n=6000, n_kv=2, n_q=8, n_needles=4, W=8, steps=2, sketch="int8",
                                  eta=1 / 16, eps=0.02, delta=0.05, n_sink=4, n_local=64, query_mode="needle_half")
    ctx = binding.VerKV(n_kv_heads=w.n_kv, n_q_heads=w.n_q, max_tokens=w.n, n_sink=w.n_sink, n_local=w.n_local,
                        eta=w.eta, seed=w.seed, sketch="int8", kv_dtype="bf16")
    kv = torch.from_numpy(w.kv_host_layout(0)).view(torch.bfloat16).pin_memory()
    obs = torch.from_numpy(np.ascontiguousarray(w.obs_q[0])).cuda()
    ctx.compress(0, 0, w.n, kv, kv.cuda(), obs, w.obs_q.shape[2], None)
    stream = torch.cuda.current_stream()
    checked_fetch = 0
    for s in range(2):
        q = torch.from_numpy(np.ascontiguousarray(w.queries[s])).cuda()
        out = torch.empty_like(q)
        ctx.decode(0, [0], q, w.eps, w.delta, out)
        trace = ctx.decode_trace(w.n_q)
        for hq in range(w.n_q):
            t = trace[hq]
            what, toks = ctx.row_weights(0, hq, w.n)
            _, _, r_all, _ = ctx.compress_state(0, 0, hq // w.group, w.n)
            w_d = torch.from_numpy(what).cuda()
            r_d = torch.from_numpy(np.ascontiguousarray(r_all[toks])).cuda()
            ref_set = ctx.exact_set(0, hq, w.n)
            results = []
            for call in range(2):
                scal = torch.full((4,), -1.0, dtype=torch.float64, device="cuda")
                kst = torch.full((1,), -1, dtype=torch.int32, device="cuda")
                ex = torch.full((len(what),), -1, dtype=torch.int32, device="cuda")
                rc = f(w_d.data_ptr(), r_d.data_ptr(), len(what), t["D"], w.eps, w.delta, scal.data_ptr(),
                       kst.data_ptr(), ex.data_ptr(), stream.cuda_stream)
                assert rc == 0, binding.STATUS.get(rc, rc)
                torch.cuda.synchronize()
                k = int(kst.item())
                results.append((scal.cpu().numpy(), k, np.sort(toks[ex[:k].cpu().numpy()])))
            for sc, k, st_set in results:
                assert abs(sc[1] - t["eps_hat"]) <= 1e-4 * abs(t["eps_hat"]) + 1e-30, (sc[1], t["eps_hat"])
                assert abs(sc[0] / t["D"] - t["beta"] / t["D"]) <= 1e-4 * abs(t["beta"] / t["D"]) + 1e-30
                assert k == t["kstar"], (k, t["kstar"])
                assert np.array_equal(st_set, ref_set)
            assert results[0][1] == results[1][1] and np.array_equal(results[0][2], results[1][2])
            checked_fetch += t["kstar"] > 0
    assert checked_fetch > 0, "no row fetched: the comparison did not exercise the ranking"
    # sizes beyond the static scratch are rejected
    big = 65536 + 1
    scal = torch.zeros(4, dtype=torch.float64, device="cuda")
    kst = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert f(scal.data_ptr(), scal.data_ptr(), big, 1.0, 0.05, 0.05, scal.data_ptr(), kst.data_ptr(),
             kst.data_ptr(), stream.cuda_stream) == 1
    ctx.close()


def _run_static(f, w_hat, r, D, eps, delta, stream, exact_fill=-7):
    """Two calls in a row on the same inputs; returns [(scalars, k*, exact indices, exact buffer)]."""
    n_l = len(w_hat)
    w_d = torch.from_numpy(np.ascontiguousarray(w_hat, np.float32)).cuda()
    r_d = torch.from_numpy(np.ascontiguousarray(r, np.float32)).cuda()
    out = []
    for call in range(2):
        scal = torch.full((4,), -1.0, dtype=torch.float64, device="cuda")
        kst = torch.full((1,), -2, dtype=torch.int32, device="cuda")
        ex = torch.full((max(n_l, 1),), exact_fill, dtype=torch.int32, device="cuda")
        rc = f(w_d.data_ptr() if n_l else 0, r_d.data_ptr() if n_l else 0, n_l, D, eps, delta, scal.data_ptr(),
               kst.data_ptr(), ex.data_ptr(), stream.cuda_stream)
        assert rc == 0, binding.STATUS.get(rc, rc)
        torch.cuda.synchronize()
        k = int(kst.item())
        exb = ex.cpu().numpy()
        out.append((scal.cpu().numpy(), k, exb[:max(k, 0)].copy(), exb))
    return out


def _against_oracle(f, w_hat, r, D_h, eps, delta, stream):
    """The oracle's decision on the same row: L tokens with sketch logits log(w_hat) (exact sketch),
    one H token carrying the rest of the denominator.  Every call's beta/D, eps_hat, k* and set must
    meet the parity bars (check_row: 1e-4 relative, the set exact up to the gain-gap exemption)."""
    n_l = len(w_hat)
    wd = np.asarray(w_hat, np.float32).astype(np.float64)
    D = float(D_h + wd.sum())
    flags = np.zeros(n_l + 1, np.uint8)
    flags[0] = 2
    r32 = np.concatenate([[1.0], r]).astype(np.float32)
    with np.errstate(divide="ignore"):
        t = np.concatenate([[math.log(D_h)], np.log(wd)])
    orow = oracle.kvfetch_row(flags, r32, t, t, eps, delta)
    verdicts = []
    for sc, k, ex, _ in _run_static(f, w_hat, r, D, eps, delta, stream):
        trace = {"beta": sc[0], "eps_hat": sc[1], "D": D, "kstar": k, "no_fetch": int(k == 0)}
        verdicts.append(check_row(trace, ex + 1, orow, eps, flags))   # token index = 1 + L index
    return orow, verdicts


def test_static_decision_matches_oracle():
    """Against the oracle: a spread of weights that fetches, a needle row, eps = 0 (every token of L is
    made exact), the largest row the static scratch takes (VERKV_STATIC_MAX_L), and lengths just past a
    power of two (the bitonic sort pads to the next one)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    f = _static_fn()
    stream = torch.cuda.current_stream()
    rng = np.random.default_rng(41)
    cases = [(6000, 1.0, 0.02, 0.05), (4097, 1.5, 0.05, 0.1), (32769, 1.0, 0.02, 0.05), (65536, 1.2, 0.01, 0.05),
             (3000, 0.8, 0.0, 0.05), (1025, 0.5, 0.3, 0.05)]
    fetched = 0
    verdict_all = []
    for n_l, sig, eps, delta in cases:
        w_hat = np.exp(sig * rng.standard_normal(n_l)).astype(np.float32)
        if n_l == 4097:
            w_hat[rng.choice(n_l, 5, replace=False)] *= 400.0   # needles
        r = rng.uniform(0.02, 0.6, n_l).astype(np.float32)
        D_h = float(w_hat.astype(np.float64).sum() * 0.05)
        orow, verdicts = _against_oracle(f, w_hat, r, D_h, eps, delta, stream)
        verdict_all += verdicts   # an exemption is returned only when check_row found it legitimate
        assert verdicts[0] == verdicts[1], (n_l, eps, verdicts)
        if eps == 0.0:
            assert orow["kstar"] == n_l
        fetched += orow["kstar"] > 0
    assert fetched >= 4
    assert verdict_all.count("ok") >= len(verdict_all) - 2, verdict_all


def test_static_decision_edge_cases():
    """n_l = 0 with eps = 0 gives k* = 0 and leaves a caller's exact buffer untouched; inputs outside the
    documented domain come back as k* = -1 with NaN scalars; sizes beyond the scratch are rejected."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    f = _static_fn()
    stream = torch.cuda.current_stream()
    for eps in (0.0, 0.05):
        for sc, k, ex, buf in _run_static(f, np.zeros(0, np.float32), np.zeros(0, np.float32), 1.0, eps, 0.05,
                                          stream, exact_fill=-7):
            assert k == 0 and np.all(buf == -7) and np.all(sc == 0.0), (eps, k, buf[:4], sc)
    # NULL exact buffer with an empty row
    scal = torch.zeros(4, dtype=torch.float64, device="cuda")
    kst = torch.full((1,), -2, dtype=torch.int32, device="cuda")
    assert f(0, 0, 0, 1.0, 0.0, 0.05, scal.data_ptr(), kst.data_ptr(), 0, stream.cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(kst.item()) == 0
    rng = np.random.default_rng(3)
    w_hat = np.exp(rng.standard_normal(500)).astype(np.float32)
    for bad_r, bad_w in [(1.0, None), (0.0, None), (None, float("inf")), (None, -1.0), (None, float("nan"))]:
        r = rng.uniform(0.1, 0.5, 500).astype(np.float32)
        wb = w_hat.copy()
        if bad_r is not None:
            r[123] = bad_r
        if bad_w is not None:
            wb[77] = bad_w
        for sc, k, ex, buf in _run_static(f, wb, r, float(w_hat.sum()) * 2, 0.01, 0.05, stream):
            assert k == -1 and np.all(np.isnan(sc)) and np.all(buf == -7), (bad_r, bad_w, k)
