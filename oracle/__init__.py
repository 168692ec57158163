"""VerKV oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.

Plain double-precision CPU restatement of "Verify Before You Fetch: Reliable
KV Cache Compression for LLM Inference" (PoissonComp: Algorithm 1, eq. (3);
KVFetch: Algorithm 2, Definition 2 / eq. (5), Lemma 1 / eq. (7), eqs. (9)-(10);
binary shrinkage: Appendix A.2; key sketch and shortlist: Appendix A.1).  The arithmetic lives in ``verkv_oracle.c``; this
module compiles it with gcc and wraps it for numpy arrays.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this module.  It imports nothing from the CUDA package.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libverkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Cert(ctypes.Structure):
    _fields_ = [("m", ctypes.c_double), ("D", ctypes.c_double), ("beta", ctypes.c_double),
                ("sum_a", ctypes.c_double), ("V", ctypes.c_double), ("b", ctypes.c_double),
                ("eps_hat", ctypes.c_double), ("n_l", ctypes.c_int64), ("kstar", ctypes.c_int64),
                ("no_fetch", ctypes.c_int32), ("pad", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "pad"}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            L = _lib
            P = ctypes.c_void_p
            i64, i32, u32, u64, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_double
            L.vko_philox4x32_10.argtypes = [P, P, P]
            L.vko_uniform.argtypes = [u64, u32, u32, u32, u32]
            L.vko_uniform.restype = ctypes.c_float
            L.vko_tau.argtypes = [i64, i32, P, i32, P, i32, i32, P]
            L.vko_waterfill.argtypes = [i64, P, i32, i32, f64, P, P, P, P]
            L.vko_waterfill.restype = i32
            L.vko_u128_to_double.argtypes = [u64, u64]
            L.vko_u128_to_double.restype = f64
            L.vko_poisson_sample.argtypes = [i64, P, u64, u32, u32, u32, P]
            L.vko_sketch_int8.argtypes = [i64, i32, P, P, P]
            L.vko_sketch_2bit.argtypes = [i64, i32, P, i32, P, P, P, P]
            L.vko_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.vko_f16_to_f32.restype = ctypes.c_float
            L.vko_logits_exact.argtypes = [i64, i32, P, P, P]
            L.vko_logits_int8.argtypes = [i64, i32, P, P, P, P]
            L.vko_logits_2bit.argtypes = [i64, i32, P, P, P, P, P, i32, P]
            L.vko_beta_breakpoints.argtypes = [i64, P, P]
            L.vko_beta_breakpoints.restype = f64
            L.vko_kvfetch_row.argtypes = [i64, P, P, P, P, f64, f64, i32, P, P, P, P, P, P]
            L.vko_kvfetch_row.restype = i32
            L.vko_kvfetch_row_ex.argtypes = [i64, P, P, P, P, P, f64, f64, i32, i32, P, P, P, P, P, P]
            L.vko_shortlist.argtypes = [i64, i32, P, P, i64, P]
            L.vko_shortlist.restype = i64
            L.vko_kvfetch_row_ex.restype = i32
            L.vko_binary_shrinkage.argtypes = [i64, P, P, P, P]
            L.vko_binary_shrinkage.restype = f64
            L.vko_attention_row.argtypes = [i64, i32, P, P, P, P, P, P, P]
            L.vko_estimate_row.argtypes = [i64, i32, P, P, P, P, P, P, f64, P]
            L.vko_estimate_row.restype = f64
            L.vko_kvfetch_rows.argtypes = [i64, i64, P, P, P, P, P, f64, f64, i32, i32, P, P, i32]
            L.vko_kvfetch_rows.restype = i32
            L.vko_num_threads.restype = i32
        return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- Philox / sample
def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().vko_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform(seed: int, token: int, kv_head: int, layer: int, seq: int) -> float:
    return lib().vko_uniform(seed, token, kv_head, layer, seq)


def poisson_sample(r32, seed: int, kv_head: int, layer: int, seq: int):
    r = _c(r32, np.float32)
    flags = np.zeros(r.shape[0], np.uint8)
    lib().vko_poisson_sample(r.shape[0], _p(r), seed, kv_head, layer, seq, _p(flags))
    return flags


# --------------------------------------------------------------------------- compress
def tau(K, Q, n_sink: int, n_local: int):
    """K [n, d], Q [rows, d] (any float dtype; values taken exactly as doubles)."""
    K = _c(K, np.float64)
    Q = _c(Q, np.float64)
    out = np.zeros(K.shape[0], np.float32)
    lib().vko_tau(K.shape[0], K.shape[1], _p(K), Q.shape[0], _p(Q), n_sink, n_local, _p(out))
    return out


def waterfill(tau32, n_sink: int, n_local: int, budget: float):
    """Returns (c, t_star, r64, r32).  Raises ValueError when the budget does not cover the forced set."""
    t = _c(tau32, np.float32)
    n = t.shape[0]
    c = ctypes.c_double()
    ts = ctypes.c_int64()
    r64 = np.zeros(n, np.float64)
    r32 = np.zeros(n, np.float32)
    rc = lib().vko_waterfill(n, _p(t), n_sink, n_local, float(budget), ctypes.byref(c), ctypes.byref(ts),
                             _p(r64), _p(r32))
    if rc != 0:
        raise ValueError("budget does not cover the sink/local tokens")
    return c.value, ts.value, r64, r32


def u128_to_double(v: int) -> float:
    return lib().vko_u128_to_double((v >> 64) & (2**64 - 1), v & (2**64 - 1))


def sketch_int8(K):
    K = _c(K, np.float32)
    n, d = K.shape
    codes = np.zeros((n, d), np.int8)
    scale = np.zeros(n, np.float32)
    lib().vko_sketch_int8(n, d, _p(K), _p(codes), _p(scale))
    return codes, scale


def sketch_2bit(K, group: int = 128):
    K = _c(K, np.float32)
    n, d = K.shape
    ng = (n + group - 1) // group
    pairs = np.zeros(d // 8, np.int32)
    codes = np.zeros((n, d // 4), np.uint8)
    zero = np.zeros((ng, d // 4), np.uint16)
    scale = np.zeros((ng, d // 4), np.uint16)
    lib().vko_sketch_2bit(n, d, _p(K), group, _p(pairs), _p(codes), _p(zero), _p(scale))
    return pairs, codes, zero, scale


def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    f = lib().vko_f16_to_f32
    return np.array([f(int(b)) for b in np.asarray(bits).ravel()], np.float32).reshape(np.shape(bits))


def kept_channels(pairs, d: int):
    pairs = np.asarray(pairs, np.int64)
    return np.concatenate([pairs, pairs + d // 2])


# --------------------------------------------------------------------------- logits
def logits_exact(q, K):
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    out = np.zeros(K.shape[0], np.float64)
    lib().vko_logits_exact(K.shape[0], K.shape[1], _p(q), _p(K), _p(out))
    return out


def logits_int8(q, codes, scale):
    q = _c(q, np.float64)
    codes = _c(codes, np.int8)
    scale = _c(scale, np.float32)
    out = np.zeros(codes.shape[0], np.float64)
    lib().vko_logits_int8(codes.shape[0], codes.shape[1], _p(q), _p(codes), _p(scale), _p(out))
    return out


def logits_2bit(q, pairs, codes, zero, scale, group: int = 128):
    q = _c(q, np.float64)
    pairs = _c(pairs, np.int32)
    codes = _c(codes, np.uint8)
    zero = _c(zero, np.uint16)
    scale = _c(scale, np.uint16)
    out = np.zeros(codes.shape[0], np.float64)
    lib().vko_logits_2bit(codes.shape[0], q.shape[0], _p(q), _p(pairs), _p(codes), _p(zero), _p(scale),
                          group, _p(out))
    return out


# --------------------------------------------------------------------------- KVFetch
def beta_breakpoints(w, r) -> float:
    w = _c(w, np.float64)
    r = _c(r, np.float64)
    return lib().vko_beta_breakpoints(w.shape[0], _p(w), _p(r))


def binary_shrinkage(w, r):
    """Appendix A.2: lambda_i in {1, r_i}.  Returns (lambda, beta, number set to r_i)."""
    w = _c(w, np.float64)
    r = _c(r, np.float64)
    lam = np.zeros(w.shape[0], np.float64)
    ns = ctypes.c_int64()
    beta = lib().vko_binary_shrinkage(w.shape[0], _p(w), _p(r), _p(lam), ctypes.byref(ns))
    return lam, beta, ns.value


def shortlist(flags, t_sketch_rows, k: int):
    """Appendix A.1 shortlist of one KV head: boolean mask of the k non-resident tokens of L with the
    largest sketch logit over the head's query rows (t_sketch_rows: [G, n]; ties: lower index)."""
    flags = _c(flags, np.uint8)
    ts = _c(t_sketch_rows, np.float64)
    G, n = ts.shape
    mask = np.zeros(n, np.uint8)
    lib().vko_shortlist(n, G, _p(flags), _p(ts), int(k), _p(mask))
    return mask.astype(bool)


def kvfetch_row(flags, r32, t_exact, t_sketch, eps: float, delta: float, mode: int = 1, shrinkage: int = 0,
                use_exact=None):
    """One query row of Algorithm 2.  Returns dict with cert scalars and arrays.
    shrinkage: 0 = the clipped coefficients of Definition 2, 1 = binary (Appendix A.2).
    use_exact: optional boolean mask of tokens of L whose exact logit replaces the sketch logit."""
    flags = _c(flags, np.uint8)
    r32 = _c(r32, np.float32)
    te = _c(t_exact, np.float64)
    ts = _c(t_sketch, np.float64)
    n = flags.shape[0]
    cert = Cert()
    lam = np.zeros(n, np.float64)
    gain = np.zeros(n, np.float64)
    n_l = int((flags != 2).sum())
    order = np.zeros(max(n_l, 1), np.int64)
    mask = np.zeros(n, np.uint8)
    resid = np.full(n_l + 1, np.nan)
    ue = None if use_exact is None else _c(np.asarray(use_exact).astype(np.uint8), np.uint8)
    lib().vko_kvfetch_row_ex(n, _p(flags), _p(r32), _p(te), _p(ts), None if ue is None else _p(ue), float(eps),
                             float(delta), int(mode), int(shrinkage), ctypes.byref(cert), _p(lam), _p(gain), _p(order),
                             _p(mask), _p(resid))
    out = cert.as_dict()
    out.update(lam=lam, gain=gain, order=order[:n_l], exact_mask=mask.astype(bool), resid=resid)
    return out


def attention_row(flags, r32, t_exact, V, lam, exact_mask):
    flags = _c(flags, np.uint8)
    r32 = _c(r32, np.float32)
    te = _c(t_exact, np.float64)
    V = _c(V, np.float64)
    lam = _c(lam, np.float64)
    mask = _c(exact_mask, np.uint8)
    out = np.zeros(V.shape[1], np.float64)
    lib().vko_attention_row(flags.shape[0], V.shape[1], _p(flags), _p(r32), _p(te), _p(V), _p(lam), _p(mask),
                            _p(out))
    return out


def estimate_row(flags, r32, t_exact, lam, exact_mask, m: float = 0.0, V=None):
    """Definition 2 / eq. (5) after the fetch: (D^, N^) with weights exp(t_exact - m); flags carry the
    sample outcome (1 = sampled).  N^ is None when V is None."""
    flags = _c(flags, np.uint8)
    r32 = _c(r32, np.float32)
    te = _c(t_exact, np.float64)
    lam = _c(lam, np.float64)
    mask = _c(exact_mask, np.uint8)
    if V is None:
        den = lib().vko_estimate_row(flags.shape[0], 0, _p(flags), _p(r32), _p(te), None, _p(lam), _p(mask),
                                     float(m), None)
        return den, None
    V = _c(V, np.float64)
    num = np.zeros(V.shape[1], np.float64)
    den = lib().vko_estimate_row(flags.shape[0], V.shape[1], _p(flags), _p(r32), _p(te), _p(V), _p(lam), _p(mask),
                                 float(m), _p(num))
    return den, num


def kvfetch_rows(flags, r32, kv_of, t_exact, t_sketch, eps, delta, mode=1, threads=0, shrinkage=0):
    """Many independent rows (OpenMP).  flags/r32: [Hkv, n]; t_*: [rows, n]."""
    flags = _c(flags, np.uint8)
    r32 = _c(r32, np.float32)
    kv_of = _c(kv_of, np.int32)
    te = _c(t_exact, np.float64)
    ts = _c(t_sketch, np.float64)
    rows, n = te.shape
    certs = (Cert * rows)()
    masks = np.zeros((rows, n), np.uint8)
    lib().vko_kvfetch_rows(rows, n, _p(flags), _p(r32), _p(kv_of), _p(te), _p(ts), float(eps), float(delta),
                           int(mode), int(shrinkage), certs, _p(masks), int(threads))
    return [c.as_dict() for c in certs], masks.astype(bool)


def num_threads() -> int:
    return lib().vko_num_threads()
