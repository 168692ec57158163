"""GPU parity: the CUDA path (through the C ABI) against the oracle on the same seeded inputs.

Bars (the spec's tolerances): bit-exact H/L membership, sample S, inclusion probabilities and
sketch codes; c, beta/D and eps_hat within 1e-4 relative; the fetched set exact except where the
oracle's gains at the k* boundary are within 1e-6 relative (or the residual certificate is within
1e-6 of eps); attention output within 2e-3 relative L2.
"""
import dataclasses
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from verified_kv_cache_gb300 import workloads

from vkcase import (GpuCase, REL_OUT, check_row, check_row_output, make_lib_ctx, oracle_compress, oracle_decode,
                    oracle_tau, rel, rel_l2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from verified_kv_cache_gb300 import build
    build.build()


def small_case(sketch, n=4000, seed=11, n_kv=2, n_q=8, steps=4, eps=0.05, delta=0.05, eta=1 / 16, batch=1,
               query_mode="needle_half"):
    w = workloads.qwen_layer_case(seed=seed, n=n, n_kv=n_kv, n_q=n_q, n_needles=4, W=8, steps=steps, sketch=sketch,
                                  eta=eta, eps=eps, delta=delta, n_sink=4, n_local=64, batch=batch,
                                  query_mode=query_mode)
    return w


CASES = {
    "tiny-exact-f32": lambda: workloads.tiny_oracle_case(),
    "int8-ragged": lambda: small_case("int8", n=4000),
    "2bit-ragged": lambda: small_case("2bit", n=4133),
    "int8-g1": lambda: small_case("int8", n=3000, n_kv=2, n_q=2),
}


def _compress_both(w, gc, b=0, tau=None):
    tau = oracle_tau(w, b) if tau is None else tau
    stats = gc.compress(b, tau=tau)
    osl = oracle_compress(w, b, tau, layer=0, seq=b)
    return tau, stats, osl


@pytest.mark.parametrize("case", list(CASES))
def test_compress_given_scores_is_bit_exact(case):
    w = CASES[case]()
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    for h in range(w.n_kv):
        c, tau_g, r, flags = ctx.compress_state(0, 0, h, w.n)
        assert np.array_equal(tau_g, np.clip(tau[h], 2.0 ** -38, 1.0))
        assert c == osl.c[h] or rel(c, osl.c[h]) <= 1e-15, (c, osl.c[h])
        assert np.array_equal(r, osl.r32[h])
        assert np.array_equal(flags, osl.flags[h])
        assert stats[h]["n_h"] == int((osl.flags[h] == 2).sum())
        assert stats[h]["n_s"] == int((osl.flags[h] == 1).sum())
        assert stats[h]["n_l"] == int((osl.flags[h] != 2).sum())
        if w.sketch == "int8":
            codes, scale = ctx.sketch_int8(0, 0, h, w.n)
            oc, osc = osl.sketch[h]
            assert np.array_equal(codes, oc) and np.array_equal(scale, osc)
        elif w.sketch == "2bit":
            pairs, codes, zero, scale = ctx.sketch_2bit(0, 0, h, w.n)
            op, oc, oz, os_ = osl.sketch[h]
            assert np.array_equal(pairs, op)
            assert np.array_equal(codes, oc) and np.array_equal(zero, oz) and np.array_equal(scale, os_)
    ctx.close()


@pytest.mark.parametrize("case", ["int8-ragged", "2bit-ragged"])
def test_importance_scores_and_end_to_end_sample(case):
    """The GPU's own scorer: tau within fp32 tolerance of the oracle's, and the sample differs only at
    threshold near-ties (c tau ~ 1 or u ~ r)."""
    w = CASES[case]()
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    gc.compress(0)
    tau_o = oracle_tau(w, 0)
    osl = oracle_compress(w, 0, tau_o)
    for h in range(w.n_kv):
        c, tau_g, r, flags = ctx.compress_state(0, 0, h, w.n)
        big = tau_o[h] > 1e-6
        assert np.allclose(tau_g[big], tau_o[h][big], rtol=2e-5, atol=0)
        assert rel(c, osl.c[h]) <= 1e-4
        bad = np.nonzero(flags != osl.flags[h])[0]
        assert len(bad) <= max(2, w.n // 1000)
        for i in bad:
            u = oracle.uniform(w.seed, int(i), h, 0, 0)
            near = abs(osl.c[h] * tau_o[h][i] - 1.0) <= 1e-4 or abs(u - osl.r32[h][i]) <= 1e-4 * osl.r32[h][i]
            assert near, (i, u, osl.r32[h][i], r[i])
    ctx.close()


def _decode_parity(w, gc, osl, eps, delta, steps=None, b=0, max_exempt_frac=0.05, shrinkage=0):
    steps = range(w.queries.shape[0]) if steps is None else steps
    ctx = gc.ctx
    counts = {"ok": 0, "exempt-b": 0, "exempt-k": 0, "exempt-g": 0}
    for s in steps:
        out = gc.decode(w.queries[s], eps, delta)
        trace = ctx.decode_trace(w.batch * w.n_q)
        rows, unions = oracle_decode(w, b, osl, w.queries[s, b], eps, delta, shrinkage=shrinkage)
        row_ok = []
        for hq in range(w.n_q):
            t = trace[b * w.n_q + hq]
            gset = ctx.exact_set(b, hq, w.n)
            verdict = check_row_output(t, gset, rows[hq], eps, out[b, hq], (s, hq))
            counts[verdict] += 1
            row_ok.append(verdict == "ok")
        for h in range(w.n_kv):
            if all(row_ok[h * w.group:(h + 1) * w.group]):
                fs = ctx.fetch_set(b, h, w.n)
                assert np.array_equal(fs, unions[h]), (s, h)
    total = sum(counts.values())
    assert counts["ok"] >= (1 - max_exempt_frac) * total, counts
    return counts


@pytest.mark.parametrize("case", list(CASES))
def test_decode_parity(case):
    w = CASES[case]()
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    _decode_parity(w, gc, osl, w.eps, w.delta)
    ctx.close()


@pytest.mark.parametrize("case", list(CASES))
def test_decode_parity_binary_shrinkage(case):
    """Appendix A.2's binary coefficients (lambda in {1, r}): the shrunk prefix of the gamma order
    (its length exact), beta, eps_hat, k*, the fetched set and the output against the oracle."""
    w = CASES[case]()
    ctx = make_lib_ctx(w, shrinkage="binary")
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    counts = _decode_parity(w, gc, osl, w.eps, w.delta, shrinkage=1)
    trace = ctx.decode_trace(w.batch * w.n_q)
    assert any(t["n_shrunk"] >= 1 for t in trace), [t["n_shrunk"] for t in trace]
    print(case, counts)
    ctx.close()


def test_binary_shrinkage_long_prefix_spans_search_levels():
    """Small inclusion probabilities make the binary prefix long (about 1 / (2 r) entries of similar
    gamma), so its end lies in a crowded bin and takes several search levels."""
    w = small_case("int8", n=12000, steps=2, query_mode="random", eta=1 / 128)
    w.queries *= 0.1   # flat weights
    ctx = make_lib_ctx(w, shrinkage="binary")
    gc = GpuCase(w, ctx)
    tau = np.full((w.n_kv, w.n), 0.5, np.float32)
    tau[:, ::7] = 0.45
    tau, stats, osl = _compress_both(w, gc, tau=tau)
    gc.decode(w.queries[0], 0.05, 0.05)
    trace = ctx.decode_trace(w.n_q)
    assert max(t["n_shrunk"] for t in trace) > 64, [t["n_shrunk"] for t in trace]
    _decode_parity(w, gc, osl, 0.05, 0.05, shrinkage=1)
    ctx.close()


@pytest.mark.parametrize("eps", [0.2, 0.01, 0.002])
def test_decode_parity_across_tolerances(eps):
    w = small_case("int8", n=6000, steps=2, query_mode="random")
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    _decode_parity(w, gc, osl, eps, 0.1)
    ctx.close()


def test_eps_zero_fetches_everything_and_matches_dense_attention():
    w = small_case("int8", n=2500, steps=2)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    for s in range(2):
        out = gc.decode(w.queries[s], 0.0, 0.05)
        trace = ctx.decode_trace(w.n_q)
        for hq in range(w.n_q):
            h = hq // w.group
            assert trace[hq]["kstar"] == stats[h]["n_l"] or trace[hq]["no_fetch"] and stats[h]["n_l"] == 0
            K = torch.tensor(w.K[0, h], dtype=torch.float64)
            V = torch.tensor(w.V[0, h], dtype=torch.float64)
            q = torch.tensor(w.queries[s, 0, hq], dtype=torch.float64)
            dense = torch.nn.functional.scaled_dot_product_attention(q[None, None, None], K[None, None],
                                                                     V[None, None])[0, 0, 0].numpy()
            assert rel_l2(out[0, hq].astype(np.float64), dense) <= REL_OUT
    ctx.close()


def test_batch_of_sequences_with_different_lengths():
    ws = [small_case("int8", n=n, seed=20 + i, steps=2) for i, n in enumerate([3000, 4100, 2049])]
    nmax = max(w.n for w in ws)
    from verified_kv_cache_gb300 import binding
    w0 = ws[0]
    ctx = binding.VerKV(n_kv_heads=w0.n_kv, n_q_heads=w0.n_q, max_tokens=nmax, n_layers=1, n_seqs=3, max_batch=3,
                        n_sink=w0.n_sink, n_local=w0.n_local, eta=w0.eta, seed=w0.seed, sketch="int8", kv_dtype="bf16")
    cases = []
    for i, w in enumerate(ws):
        gc = GpuCase(w, ctx)
        tau = oracle_tau(w, 0)
        gc.compress(0, seq=i, tau=tau)
        cases.append((gc, oracle_compress(w, 0, tau, layer=0, seq=i)))
    for s in range(2):
        q = np.stack([w.queries[s, 0] for w in ws])          # [3, Hq, d]
        qt = torch.from_numpy(q).cuda()
        out = torch.empty_like(qt)
        ctx.decode(0, [0, 1, 2], qt, ws[0].eps, ws[0].delta, out)
        torch.cuda.synchronize()
        out = out.cpu().numpy()
        trace = ctx.decode_trace(3 * w0.n_q)
        for i, w in enumerate(ws):
            rows, unions = oracle_decode(w, 0, cases[i][1], w.queries[s, 0], w.eps, w.delta)
            for hq in range(w.n_q):
                check_row_output(trace[i * w.n_q + hq], ctx.exact_set(i, hq, w.n), rows[hq], w.eps, out[i, hq],
                                 (s, i, hq))
    ctx.close()


def test_large_kstar_on_the_cluster_path():
    """Flat attention and a tight tolerance: k* runs into the thousands (well past any fixed candidate
    width), decided by the cluster kernel's radix search, and matches the oracle."""
    w = small_case("int8", n=20000, steps=1, query_mode="random", eta=1 / 8)
    w.queries *= 0.3
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    eps = 0.002
    gc.decode(w.queries[0], eps, 0.05)
    trace = ctx.decode_trace(w.n_q)
    assert max(t["kstar"] for t in trace) > 8192, [t["kstar"] for t in trace]
    _decode_parity(w, gc, osl, eps, 0.05, steps=[0])
    ctx.close()


def test_full_row_path_for_long_rows():
    """|L| above the fused decision's limit (262144 entries per row) uses the multi-kernel path: on-chip
    ranking of 4096 candidates and, when k* lies beyond them, the full-row sort."""
    w = small_case("int8", n=280000, steps=1, query_mode="random", eta=1 / 16, n_kv=2, n_q=4)
    w.queries *= 0.3
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc, tau=workloads.synthetic_scores(w.n_kv, w.n, seed=9))
    assert max(s["n_l"] for s in stats) > 262144
    eps = 0.005
    gc.decode(w.queries[0], eps, 0.05)
    trace = ctx.decode_trace(w.n_q)
    assert any(t["fallback"] for t in trace), [t["kstar"] for t in trace]
    _decode_parity(w, gc, osl, eps, 0.05, steps=[0])
    ctx.close()


@pytest.mark.parametrize("shrinkage", ["clipped", "binary"])
def test_streaming_decision_on_rows_beyond_shared_memory(shrinkage):
    """Rows longer than the on-chip decision holds (16 x 8192 entries): the streaming variant of the
    fused decision (entries re-read from L2 in every pass), with both coefficient rules.  n = 250000
    gives |L| of about 234000 per row; binary shrinkage runs there too."""
    w = small_case("int8", n=250000, steps=2, query_mode="needle_half", eta=1 / 16, n_kv=2, n_q=4)
    ctx = make_lib_ctx(w, shrinkage=shrinkage)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc, tau=workloads.synthetic_scores(w.n_kv, w.n, seed=19))
    assert max(s["n_l"] for s in stats) > 131072
    for eps in (0.05, 0.01):
        counts = _decode_parity(w, gc, osl, eps, 0.05, shrinkage=1 if shrinkage == "binary" else 0)
        trace = ctx.decode_trace(w.n_q)
        assert not any(t["fallback"] for t in trace)
        print(shrinkage, eps, counts)
    ctx.close()


def test_streaming_and_on_chip_decisions_agree():
    """The same sequence decoded alone (one wave: the on-chip decision) and as eight copies in one call
    (256 query rows: the streaming decision).  Both must meet the oracle's bars on every row; k* and
    the sets agree except at near-ties, which the oracle comparison exempts row by row."""
    base = small_case("int8", n=6000, steps=2, query_mode="needle_half", n_kv=8, n_q=32)
    w8 = dataclasses.replace(base, batch=8, K=np.repeat(base.K, 8, axis=0), V=np.repeat(base.V, 8, axis=0),
                             obs_q=np.repeat(base.obs_q, 8, axis=0), queries=np.repeat(base.queries, 8, axis=1))
    ctx = make_lib_ctx(w8)
    gc = GpuCase(w8, ctx)
    tau = oracle_tau(base, 0)
    slots = []
    for b in range(8):
        gc.compress(b, seq=b, tau=tau)
        slots.append(oracle_compress(w8, b, tau, layer=0, seq=b))
    for s in range(2):
        single = gc.decode(w8.queries[s, :1], w8.eps, w8.delta, seq_ids=[0])     # on-chip
        tr1 = ctx.decode_trace(w8.n_q)
        sets1 = [ctx.exact_set(0, hq, w8.n) for hq in range(w8.n_q)]
        full = gc.decode(w8.queries[s], w8.eps, w8.delta)                         # streaming
        tr8 = ctx.decode_trace(8 * w8.n_q)
        for b in range(8):
            rows, _ = oracle_decode(w8, b, slots[b], w8.queries[s, b], w8.eps, w8.delta)
            for hq in range(w8.n_q):
                check_row_output(tr8[b * w8.n_q + hq], ctx.exact_set(b, hq, w8.n), rows[hq], w8.eps, full[b, hq],
                                 (s, b, hq))
        rows0, _ = oracle_decode(w8, 0, slots[0], w8.queries[s, 0], w8.eps, w8.delta)
        for hq in range(w8.n_q):
            check_row_output(tr1[hq], sets1[hq], rows0[hq], w8.eps, single[0, hq], (s, "single", hq))
    ctx.close()


def test_decode_is_deterministic():
    w = small_case("2bit", n=4133, steps=2)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    _compress_both(w, gc)
    a = gc.decode(w.queries[1], w.eps, w.delta)
    sa = [ctx.exact_set(0, h, w.n) for h in range(w.n_q)]
    b = gc.decode(w.queries[1], w.eps, w.delta)
    sb = [ctx.exact_set(0, h, w.n) for h in range(w.n_q)]
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert all(np.array_equal(x, y) for x, y in zip(sa, sb))
    ctx.close()


def test_decode_before_compress_and_bad_arguments_are_rejected():
    from verified_kv_cache_gb300 import binding
    w = small_case("int8", n=2000, steps=1)
    ctx = make_lib_ctx(w)
    q = torch.zeros(1, w.n_q, w.d, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(binding.VerkvError) as e:
        ctx.decode(0, [0], q, 0.05, 0.05, out)
    assert e.value.status == 6
    gc = GpuCase(w, ctx)
    gc.compress(0, tau=oracle_tau(w, 0))
    for eps, delta in [(-1.0, 0.05), (0.05, 0.0), (0.05, 1.0), (float("nan"), 0.1)]:
        with pytest.raises(binding.VerkvError) as e:
            ctx.decode(0, [0], q, eps, delta, out)
        assert e.value.status == 1
    ctx.close()


def test_qwen_layer_full_size_binary_shrinkage():
    """The Qwen3-4B-shaped 32K-token layer with the 2-bit sketch and binary coefficients."""
    w = workloads.qwen_layer_case(sketch="2bit", steps=2)
    ctx = make_lib_ctx(w, shrinkage="binary")
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    counts = _decode_parity(w, gc, osl, w.eps, w.delta, steps=range(2), shrinkage=1)
    print(counts)
    ctx.close()


def test_importance_scores_full_size():
    """The GPU's own importance scorer (tensor cores) at the Qwen3-4B-shaped layer's shape: n = 32768,
    GQA 32/8, 32 observation queries per query head (128 observation rows per KV head), bf16 keys.
    tau within fp32 tolerance of the oracle's, c within 1e-4, and the end-to-end sample equal to the
    oracle's except at threshold near-ties."""
    w = workloads.qwen_layer_case(sketch="2bit", steps=1)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    gc.compress(0)
    tau_o = oracle_tau(w, 0)
    osl = oracle_compress(w, 0, tau_o)
    n_bad = 0
    for h in range(w.n_kv):
        c, tau_g, r, flags = ctx.compress_state(0, 0, h, w.n)
        big = tau_o[h] > 1e-6
        assert big.sum() > 100
        assert np.allclose(tau_g[big], tau_o[h][big], rtol=2e-5, atol=0), h
        assert np.all(np.abs(tau_g[~big] - tau_o[h][~big]) <= 1e-10), h
        assert rel(c, osl.c[h]) <= 1e-4
        bad = np.nonzero(flags != osl.flags[h])[0]
        n_bad += len(bad)
        for i in bad:
            u = oracle.uniform(w.seed, int(i), h, 0, 0)
            near = abs(osl.c[h] * tau_o[h][i] - 1.0) <= 1e-4 or abs(u - osl.r32[h][i]) <= 1e-4 * osl.r32[h][i]
            assert near, (h, i, u, osl.r32[h][i], r[i])
    assert n_bad <= 8, n_bad
    ctx.close()


def test_qwen_layer_full_size_warm_staging_cache():
    """The bench's state: the Qwen3-4B-shaped 32K layer (2-bit sketch) decoded for all 64 steps in
    order, so that by the last steps most fetched rows come from the staging cache.  Steps 0-3 and
    60-63 are checked row by row against the oracle (every row's output included); the steps between
    only warm the cache."""
    w = workloads.qwen_layer_case(sketch="2bit", steps=64)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    _decode_parity(w, gc, osl, w.eps, w.delta, steps=range(4))
    for s in range(4, 60):
        gc.decode(w.queries[s], w.eps, w.delta)
    nu = nh = 0
    counts = _decode_parity(w, gc, osl, w.eps, w.delta, steps=range(60, 64))
    for s in (61, 63):   # random queries: they fetch; most of their rows are staged by now
        gc.decode(w.queries[s], w.eps, w.delta)
        for h in range(w.n_kv):
            u, hr = ctx.fetch_stats(0, h)
            nu += u
            nh += hr
    assert nu > 0 and 0 < nh < nu, (nu, nh)   # the bounded cache is full: some rows staged, the rest fetched
    print(counts, "rows needed", nu, "over the link", nh)
    ctx.close()


@pytest.mark.parametrize("sketch", ["2bit", "int8"])
def test_qwen_layer_full_size(sketch):
    """The Qwen3-4B-shaped 32K-token layer (GQA 32/8) at full size, first decode steps, every row."""
    w = workloads.qwen_layer_case(sketch=sketch, steps=4)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    counts = _decode_parity(w, gc, osl, w.eps, w.delta, steps=range(4))
    print(sketch, counts)
    ctx.close()


@pytest.mark.parametrize("sketch", ["int8", "2bit", "exact"])
def test_gqa8_group(sketch):
    """Eight query heads per KV head (the widest group built): the int8 scorer's tensor-core tile is
    N = 32 (24 query pieces), the 2-bit and exact scorers their G = 8 variants."""
    w = small_case(sketch, n=5000, n_kv=2, n_q=16, steps=2)
    if sketch == "exact":
        w.sketch = "exact"
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    _decode_parity(w, gc, osl, w.eps, w.delta)
    ctx.close()


def test_batch_32_sequences():
    """The largest batch built (32 sequences in one call), ragged lengths."""
    from verified_kv_cache_gb300 import binding
    B = 32
    ws = [small_case("int8", n=1500 + 37 * i, seed=200 + i, steps=1, n_kv=2, n_q=8) for i in range(B)]
    nmax = max(w.n for w in ws)
    w0 = ws[0]
    ctx = binding.VerKV(n_kv_heads=w0.n_kv, n_q_heads=w0.n_q, max_tokens=nmax, n_layers=1, n_seqs=B, max_batch=B,
                        n_sink=w0.n_sink, n_local=w0.n_local, eta=w0.eta, seed=w0.seed, sketch="int8", kv_dtype="bf16")
    slots, cases = [], []   # the cases own the pinned host K/V the library borrows until release
    for i, w in enumerate(ws):
        gc = GpuCase(w, ctx)
        tau = oracle_tau(w, 0)
        gc.compress(0, seq=i, tau=tau)
        cases.append(gc)
        slots.append(oracle_compress(w, 0, tau, layer=0, seq=i))
    q = np.stack([w.queries[0, 0] for w in ws])
    qt = torch.from_numpy(q).cuda()
    out = torch.empty_like(qt)
    ctx.decode(0, list(range(B)), qt, w0.eps, w0.delta, out)
    torch.cuda.synchronize()
    out = out.cpu().numpy()
    trace = ctx.decode_trace(B * w0.n_q)
    ok = 0
    for i, w in enumerate(ws):
        rows, unions = oracle_decode(w, 0, slots[i], w.queries[0, 0], w.eps, w.delta)
        for hq in range(w.n_q):
            v = check_row_output(trace[i * w.n_q + hq], ctx.exact_set(i, hq, w.n), rows[hq], w.eps, out[i, hq],
                                 (i, hq))
            ok += v == "ok"
    assert ok >= 0.95 * B * w0.n_q
    ctx.close()


def test_eta_one_keeps_every_token():
    """eta = 1: every token has r = 1, L is empty, nothing is fetched and the output is the dense
    softmax attention."""
    w = small_case("int8", n=1000, steps=2, eta=1.0)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    assert all(s["n_l"] == 0 and s["n_h"] == w.n for s in stats)
    for s in range(2):
        out = gc.decode(w.queries[s], w.eps, w.delta)
        trace = ctx.decode_trace(w.n_q)
        for hq in range(w.n_q):
            h = hq // w.group
            assert trace[hq]["n_l"] == 0 and trace[hq]["kstar"] == 0 and trace[hq]["no_fetch"] == 1
            assert trace[hq]["eps_hat"] == 0.0
            K = torch.tensor(w.K[0, h], dtype=torch.float64)
            V = torch.tensor(w.V[0, h], dtype=torch.float64)
            qq = torch.tensor(w.queries[s, 0, hq], dtype=torch.float64)
            dense = torch.nn.functional.scaled_dot_product_attention(qq[None, None, None], K[None, None],
                                                                     V[None, None])[0, 0, 0].numpy()
            assert rel_l2(out[0, hq].astype(np.float64), dense) <= REL_OUT
        for h in range(w.n_kv):
            assert len(ctx.fetch_set(0, h, w.n)) == 0
    ctx.close()


def test_smallest_context():
    """n = sink + local + 3: three tokens share the budget left after the forced windows."""
    w = workloads.qwen_layer_case(seed=13, n=4 + 64 + 3, n_kv=2, n_q=8, n_needles=0, W=8, steps=2, sketch="int8",
                                  eta=0.98, eps=0.05, delta=0.05, n_sink=4, n_local=64, query_mode="random")
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    _decode_parity(w, gc, osl, w.eps, w.delta)
    _decode_parity(w, gc, osl, 0.0, w.delta)   # eps = 0: the whole of L is made exact
    ctx.close()


@pytest.mark.parametrize("sketch", ["int8", "2bit", "exact"])
def test_appended_tokens_join_h(sketch):
    """Decode-time growth (App. A.3.1: the resident list grows as tokens are generated): tokens
    appended after compress are H -- exact logits, in D_cert, attended with weight 1 -- while the
    prefix's L, S, r and sketch stay as compressed.  Appends of 1 (from pinned host memory), 1 and 298
    tokens (device memory), a decode after each; the last step's queries point at an appended token.  Against the oracle run on the prefix's
    compress state with the appended tokens flagged H."""
    n0, t = 4000, 300
    full = small_case(sketch, n=n0 + t, steps=3)
    w0 = dataclasses.replace(full, n=n0, K=full.K[:, :, :n0].copy(), V=full.V[:, :, :n0].copy())
    rng = np.random.default_rng(23)
    qs = full.queries.copy()
    for hq in range(full.n_q):   # step 2: every query row near appended token n0 + 100 of its KV head
        qs[2, 0, hq] = 3.0 * full.K[0, hq // full.group, n0 + 100] + rng.standard_normal(full.d)
    ctx = make_lib_ctx(w0, max_tokens=n0 + t)
    ctx.set_append_capacity(t)
    gc = GpuCase(w0, ctx)
    tau, stats, osl = _compress_both(w0, gc)
    tail = full.kv_host_layout(0)[:, n0:]
    counts = {"ok": 0, "exempt": 0}
    done = 0
    for s, m in enumerate([1, 1, t - 2]):
        piece = torch.from_numpy(np.ascontiguousarray(tail[:, done:done + m]))
        if full.kv_dtype == "bf16":
            piece = piece.view(torch.bfloat16)
        piece = piece.pin_memory() if s == 0 else piece.to("cuda")   # pinned host rows, then device rows
        ctx.append(0, 0, m, piece)
        done += m
        assert ctx.appended(0, 0) == done
        cur = dataclasses.replace(full, n=n0 + done, K=full.K[:, :, :n0 + done], V=full.V[:, :, :n0 + done])
        out = gc.decode(qs[s], full.eps, full.delta)
        trace = ctx.decode_trace(full.n_q)
        rows, _ = oracle_decode(cur, 0, osl, qs[s, 0], full.eps, full.delta)
        for hq in range(full.n_q):
            v = check_row_output(trace[hq], ctx.exact_set(0, hq, cur.n), rows[hq], full.eps, out[0, hq], (s, hq))
            counts["ok" if v == "ok" else "exempt"] += 1
    assert counts["ok"] >= 0.9 * sum(counts.values()), counts
    # the step aimed at an appended token attends mostly to it: the output is near its value row
    for hq in range(full.n_q):
        assert rel_l2(out[0, hq].astype(np.float64), full.V[0, hq // full.group, n0 + 100]) < 0.1, hq
    with pytest.raises(binding_error()):
        ctx.append(0, 0, 1, piece)   # beyond the room reserved at compress
    gc.compress(0, tau=tau)          # a new compress drops the appended tokens
    assert ctx.appended(0, 0) == 0
    print(sketch, counts)
    ctx.close()


def binding_error():
    from verified_kv_cache_gb300 import binding
    return binding.VerkvError


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """Failure detection without a GPU fault: a kernel whose bounded mbarrier wait is given nothing to
    wait for gives up, raises the context's error word, and the call reports VERKV_ETIMEOUT; the next
    decode of the same context runs and returns the same output as before."""
    w = small_case("int8", n=3000, steps=2)
    ctx = make_lib_ctx(w)
    gc = GpuCase(w, ctx)
    _compress_both(w, gc)
    before = gc.decode(w.queries[1], w.eps, w.delta)
    assert ctx.selftest_wait_timeout() == 4   # VERKV_ETIMEOUT
    assert ctx.selftest_wait_timeout() == 4   # the word was cleared by the report and raised again
    after = gc.decode(w.queries[1], w.eps, w.delta)
    assert np.array_equal(before, after)
    ctx.close()


def test_staging_cache_reuses_fetched_rows():
    """Rows fetched over the host link are staged in device memory and read from there by later
    decodes of the slot: repeating a decode moves no row over the link and gives bit-identical
    outputs; with staging off every needed row crosses the link each time; a capacity of k rows per
    KV head keeps the first k fetched, the default ceil(eta n) of them.  The outputs never depend on the
    setting."""
    w = small_case("int8", n=6000, steps=2, query_mode="random")
    outs = {}
    eta_n = math.ceil(w.eta * w.n)
    for cap in [-1, 0, 10, -2]:
        ctx = make_lib_ctx(w)
        ctx.set_stage_capacity(cap)
        ctx.set_prefetch(0)   # every needed row not staged crosses the host link (the prefetch has its own test)
        gc = GpuCase(w, ctx)
        tau, stats, osl = _compress_both(w, gc)
        first = gc.decode(w.queries[0], 0.01, 0.05)
        s1 = [ctx.fetch_stats(0, h) for h in range(w.n_kv)]
        assert all(nu > 0 and nh == nu for nu, nh in s1), s1
        second = gc.decode(w.queries[0], 0.01, 0.05)
        s2 = [ctx.fetch_stats(0, h) for h in range(w.n_kv)]
        assert [nu for nu, _ in s2] == [nu for nu, _ in s1]
        for (nu, nh) in s2:
            expect = {-1: 0, 0: nu, 10: nu - min(10, nu), -2: nu - min(eta_n, nu)}[cap]
            assert nh == expect, (cap, nu, nh)
        assert np.array_equal(first.view(np.uint32), second.view(np.uint32))
        outs[cap] = first
        if cap == -1:
            _decode_parity(w, gc, osl, 0.01, 0.05)   # both steps, the second partly from the cache
        ctx.close()
    assert np.array_equal(outs[-1].view(np.uint32), outs[0].view(np.uint32))
    assert np.array_equal(outs[-1].view(np.uint32), outs[10].view(np.uint32))
    assert np.array_equal(outs[-1].view(np.uint32), outs[-2].view(np.uint32))


def test_prefetch_copies_ahead_and_changes_no_result():
    """The speculative prefetch copies rows of likely-fetched tokens while the decision runs; the
    attention reads the needed ones from its buffer.  Outputs and exact sets are bit-identical with it
    on and off; with staging off, every needed row comes either from the buffer or over the host link
    (n_host + n_used = n_union), the buffer serves only rows it holds (n_used <= n_copied <= cap), and
    on random queries it serves some.  Parity against the oracle with the prefetch on runs in every
    other test (it is on by default)."""
    w = small_case("int8", n=8000, steps=4, query_mode="needle_half")
    res = {}
    for pf in (0, 512):
        ctx = make_lib_ctx(w)
        ctx.set_stage_capacity(0)
        ctx.set_prefetch(pf)
        gc = GpuCase(w, ctx)
        tau, stats, osl = _compress_both(w, gc)
        outs, sets, st_ = [], [], []
        for s in range(4):
            outs.append(gc.decode(w.queries[s], 0.01, 0.05))
            sets.append([ctx.exact_set(0, hq, w.n) for hq in range(w.n_q)])
            st_.append([(ctx.fetch_stats(0, h), ctx.prefetch_stats(0, h)) for h in range(w.n_kv)])
        if pf:
            _decode_parity(w, gc, osl, 0.01, 0.05)
        res[pf] = (outs, sets, st_)
        ctx.close()
    for s in range(4):
        assert np.array_equal(res[0][0][s].view(np.uint32), res[512][0][s].view(np.uint32)), s
        assert all(np.array_equal(x, y) for x, y in zip(res[0][1][s], res[512][1][s]))
        for ((nu0, nh0), (nc0, nd0)), ((nu, nh), (nc, nd)) in zip(res[0][2][s], res[512][2][s]):
            assert nc0 == 0 and nd0 == 0 and nh0 == nu0
            assert nu == nu0 and nh + nd == nu and nd <= nc <= 512, (s, nu, nh, nc, nd)
    used = sum(nd for s in (1, 3) for (_, (nc, nd)) in res[512][2][s])
    assert used > 0, res[512][2]


def test_call_timeline_orders_the_kernels_and_changes_no_result():
    """verkv_set_timeline records, per decode call, when the decision, the prefetch and the attention
    started and ended (device times after the scoring kernel started).  The entries follow the launch
    order (the decision waits for the scoring, the attention for the decision and the prefetch), every
    time lies within the call, and the outputs are bit-identical with recording on and off."""
    from verified_kv_cache_gb300 import binding
    w = small_case("int8", n=8000, steps=4, query_mode="needle_half")
    outs = {}
    for on in (False, True):
        ctx = make_lib_ctx(w)
        ctx.set_timeline(on)
        gc = GpuCase(w, ctx)
        _compress_both(w, gc)
        outs[on] = []
        for s in range(4):
            outs[on].append(gc.decode(w.queries[s], 0.01, 0.05))
            if on:
                t = ctx.timeline()
                assert all(np.isfinite(t[k]) for k in ("decide_start", "decide_end", "attn_start", "attn_end")), t
                assert 0.0 <= t["decide_start"] <= t["decide_end"] <= t["attn_start"] <= t["attn_end"] < 1e6, t
                if np.isfinite(t["prefetch_start"]):
                    assert t["prefetch_start"] <= t["prefetch_binned"] <= t["prefetch_end"] <= t["attn_start"], t
            else:
                with pytest.raises(binding.VerkvError):
                    ctx.timeline()
        ctx.close()
    for s in range(4):
        assert np.array_equal(outs[False][s].view(np.uint32), outs[True][s].view(np.uint32)), s


def _shortlist_near_tie(orow, got_tokens):
    """The device shortlist may differ from the oracle's only where the oracle's scores of the
    differing tokens lie within 1e-6 (relative) of the score at the shortlist boundary."""
    want = np.nonzero(orow["shortlist"])[0]
    diff = np.setxor1d(want, got_tokens)
    if len(diff) == 0:
        return True
    sc = orow["sl_score"]
    edge = sc[want].min() if len(want) else 0.0
    return bool(np.all(np.abs(sc[diff] - edge) <= 1e-6 * max(abs(edge), 1e-30)))


@pytest.mark.parametrize("pool,n", [(1, 6000), (2, 6000), (24, 6000), (0, 180)])
def test_shortlist_ties_and_short_rows(pool, n):
    """Appendix A.1's shortlist where sketch scores tie exactly: every key is a copy of one of `pool`
    rows, so equal scores are bit-equal on both sides and the k-th largest is broken by token order
    (exact set match, no exemption).  pool 1 and 2 put thousands of keys at the boundary value, pool 24
    a few hundred; pool 0 keeps the keys and makes L minus S shorter than the shortlist (all taken)."""
    w = small_case("int8", n=n, steps=2, eta=1 / 16 if pool else 0.5)
    if pool:
        rng = np.random.default_rng(5)
        for b in range(w.batch):
            for h in range(w.n_kv):
                rows = rng.standard_normal((pool, w.d)).astype(np.float32)
                w.K[b, h] = rows[np.arange(w.n) % pool]
    ctx = make_lib_ctx(w)
    ctx.set_shortlist(128)
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    for s in range(w.queries.shape[0]):
        gc.decode(w.queries[s], w.eps, w.delta)
        rows, _ = oracle_decode(w, 0, osl, w.queries[s, 0], w.eps, w.delta, shortlist=128)
        for h in range(w.n_kv):
            got = ctx.shortlist(0, h)
            want = np.nonzero(rows[h * w.group]["shortlist"])[0]
            n_cand = int((osl.flags[h] == 0).sum())
            assert len(want) == min(128, n_cand)
            if pool == 0:
                assert n_cand <= 128
            assert np.array_equal(got, want), (pool, s, h, np.setxor1d(got, want)[:8])
    ctx.close()


def _oracle_row_with_shortlist(orow, tokens, eps, delta, shrinkage):
    """The oracle's decision of a row, re-run with the DEVICE's shortlist (a legitimate near-tie
    choice at the shortlist boundary): exact weights for the sampled tokens and those tokens."""
    flags, r32, te, ts, V = orow["_flags"], orow["_r32"], orow["_te"], orow["_ts"], orow["_V"]
    sl = np.zeros(len(flags), bool)
    sl[np.asarray(tokens, np.int64)] = True
    use = sl | (flags == 1)
    res = oracle.kvfetch_row(flags, r32, te, ts, eps, delta, shrinkage=shrinkage, use_exact=use)
    if shrinkage == 1:
        Lm = flags != 2
        res["w_l"] = np.exp(np.where(use, te, ts)[Lm] - res["m"])
        res["r_l"] = r32[Lm].astype(np.float64)
        res["n_shrunk"] = int((res["lam"][Lm] < 1.0).sum())
    res["out"] = oracle.attention_row(flags, r32, te, V, res["lam"], res["exact_mask"])
    res["_flags"], res["_r32"], res["_te"], res["_ts"], res["_V"] = flags, r32, te, ts, V
    return res


@pytest.mark.parametrize("sketch,shrinkage,shape", [("int8", "clipped", "g4"), ("2bit", "clipped", "g4"),
                                                    ("2bit", "binary", "g4"), ("int8", "clipped", "g8"),
                                                    ("exact", "clipped", "tiny")])
def test_shortlist_parity(sketch, shrinkage, shape):
    """Appendix A.1's deployed certificate weights: the shortlist of 128 tokens per KV head (exact set
    match, near-ties exempt) and exact weights for sampled and shortlisted tokens in the decision;
    beta, eps_hat, k*, the fetched set and the output against the oracle run with the same weights."""
    if shape == "tiny":      # fp32 K/V, one query head per KV head, exact sketch
        w = workloads.tiny_oracle_case()
    elif shape == "g8":
        w = small_case(sketch, n=6000, n_kv=2, n_q=16, steps=4)
    else:
        w = small_case(sketch, n=6000, steps=4)
    ctx = make_lib_ctx(w, shrinkage=shrinkage)
    ctx.set_shortlist(128)
    sh = 1 if shrinkage == "binary" else 0
    gc = GpuCase(w, ctx)
    tau, stats, osl = _compress_both(w, gc)
    counts = {"ok": 0, "exempt": 0}
    for s in range(w.queries.shape[0]):
        out = gc.decode(w.queries[s], w.eps, w.delta)
        trace = ctx.decode_trace(w.n_q)
        rows, unions = oracle_decode(w, 0, osl, w.queries[s, 0], w.eps, w.delta, shortlist=128, shrinkage=sh)
        for h in range(w.n_kv):
            got = ctx.shortlist(0, h)
            orow = rows[h * w.group]
            assert len(got) == min(128, int((osl.flags[h] == 0).sum()))
            same = np.array_equal(got, np.nonzero(orow["shortlist"])[0])
            assert same or _shortlist_near_tie(orow, got), (s, h)
            for g in range(w.group):
                hq = h * w.group + g
                orow_g = rows[hq] if same else _oracle_row_with_shortlist(rows[hq], got, w.eps, w.delta, sh)
                v = check_row_output(trace[hq], ctx.exact_set(0, hq, w.n), orow_g, w.eps, out[0, hq], (s, hq))
                counts["ok" if v == "ok" and same else "exempt"] += 1
    assert counts["ok"] >= 0.9 * sum(counts.values()), counts
    print(sketch, shrinkage, shape, counts)
    ctx.close()
