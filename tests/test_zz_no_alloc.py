"""The allocation-free certificate entry point, verkv_certify_row_static.

It exists for callers that cannot allocate device memory: code running inside a CUDA stream capture
whose graph must not own allocations, or under a fixed external memory budget where cudaMalloc is
unavailable.  It takes one query row's sketch weights and inclusion probabilities and returns beta,
eps_hat, k* and the tokens to make exact, using a static device array as its only scratch.

Checked here through the C ABI against the decision verkv_decode makes for the same rows (the
existing entry point), on two calls in a row (the static scratch keeps the previous call's contents).
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from verified_kv_cache_gb300 import binding, build, workloads

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
