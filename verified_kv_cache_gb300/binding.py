"""Thin ctypes binding over libverkv.so (include/verkv.h).  Argument marshalling only: every step of
the path runs in the library's CUDA kernels.  Raises if the library has not been built; there is
no fallback implementation."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB
HEADER = os.path.join(_build.ROOT, "include", "verkv.h")

SKETCH = {"exact": 0, "int8": 1, "2bit": 2}
DTYPE = {"bf16": 0, "f32": 1}
SHRINKAGE = {"clipped": 0, "binary": 1}
STATUS = {0: "VERKV_OK", 1: "VERKV_EINVAL", 2: "VERKV_ENOMEM", 3: "VERKV_ECUDA", 4: "VERKV_ETIMEOUT",
          5: "VERKV_EUNSUPPORTED", 6: "VERKV_ESTATE"}


class VerkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


STAGE_ETA_N = -2   # default staging capacity: ceil(eta n) rows per KV head
STAGE_ALL = -1     # room for every row of L minus S


class Config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_seqs", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("n_sink", ctypes.c_int32), ("n_local", ctypes.c_int32),
                ("sketch_group", ctypes.c_int32), ("shrinkage", ctypes.c_int32),
                ("eta", ctypes.c_double), ("seed", ctypes.c_uint64), ("sketch", ctypes.c_int),
                ("kv_dtype", ctypes.c_int)]


class HeadStats(ctypes.Structure):
    _fields_ = [("c", ctypes.c_double), ("n_capped", ctypes.c_int32), ("n_h", ctypes.c_int32),
                ("n_l", ctypes.c_int32), ("n_s", ctypes.c_int32), ("n_resident", ctypes.c_int32),
                ("pad", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "pad"}


class RowTrace(ctypes.Structure):
    _fields_ = [("m", ctypes.c_double), ("D", ctypes.c_double), ("beta", ctypes.c_double),
                ("sum_a", ctypes.c_double), ("V", ctypes.c_double), ("b", ctypes.c_double),
                ("eps_hat", ctypes.c_double), ("n_l", ctypes.c_int32), ("kstar", ctypes.c_int32),
                ("no_fetch", ctypes.c_int32), ("fallback", ctypes.c_int32), ("n_fetch", ctypes.c_int32),
                ("beta_iters", ctypes.c_int32), ("sel_passes", ctypes.c_int32), ("phase_ns", ctypes.c_uint32 * 6),
                ("n_shrunk", ctypes.c_int32)]

    def as_dict(self):
        d = {k: getattr(self, k) for k, _ in self._fields_ if k != "phase_ns"}
        d["phase_ns"] = list(self.phase_ns)
        return d


_lib = None


def declared_functions() -> list[str]:
    """Names of the functions include/verkv.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(verkv_[a-z0-9_]+)\s*\(", text)))


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m verified_kv_cache_gb300.build` "
                           "(the library has no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_double
    st = ctypes.c_int
    L.verkv_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(P)]
    L.verkv_create.restype = st
    L.verkv_destroy.argtypes = [P]
    L.verkv_destroy.restype = st
    L.verkv_compress.argtypes = [P, i32, i32, i32, P, P, P, i32, P, P, P]
    L.verkv_compress.restype = st
    L.verkv_decode.argtypes = [P, i32, P, i32, P, f64, f64, P, P]
    L.verkv_decode.restype = st
    L.verkv_release.argtypes = [P, i32, i32]
    L.verkv_release.restype = st
    L.verkv_get_compress_state.argtypes = [P, i32, i32, i32, P, P, P, P, P]
    L.verkv_get_compress_state.restype = st
    L.verkv_get_sketch.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P]
    L.verkv_get_sketch.restype = st
    L.verkv_get_decode_trace.argtypes = [P, P, i32, P]
    L.verkv_get_decode_trace.restype = st
    L.verkv_get_exact_set.argtypes = [P, i32, i32, P, i32, P, P]
    L.verkv_get_exact_set.restype = st
    L.verkv_get_fetch_set.argtypes = [P, i32, i32, P, i32, P, P]
    L.verkv_get_fetch_set.restype = st
    L.verkv_get_fetch_stats.argtypes = [P, i32, i32, P, P, P]
    L.verkv_get_fetch_stats.restype = st
    L.verkv_set_shortlist.argtypes = [P, i32]
    L.verkv_set_shortlist.restype = st
    L.verkv_get_shortlist.argtypes = [P, i32, i32, P, i32, P, P]
    L.verkv_get_shortlist.restype = st
    L.verkv_set_stage_capacity.argtypes = [P, ctypes.c_int64]
    L.verkv_set_stage_capacity.restype = st
    L.verkv_set_prefetch.argtypes = [P, i32]
    L.verkv_set_prefetch.restype = st
    L.verkv_get_prefetch_stats.argtypes = [P, i32, i32, P, P, P]
    L.verkv_get_prefetch_stats.restype = st
    L.verkv_set_timeline.argtypes = [P, i32]
    L.verkv_set_timeline.restype = st
    L.verkv_get_timeline.argtypes = [P, P, P]
    L.verkv_get_timeline.restype = st
    L.verkv_selftest_wait_timeout.argtypes = [P, P]
    L.verkv_selftest_wait_timeout.restype = st
    L.verkv_set_append_capacity.argtypes = [P, i32]
    L.verkv_set_append_capacity.restype = st
    L.verkv_append.argtypes = [P, i32, i32, i32, P, P]
    L.verkv_append.restype = st
    L.verkv_get_appended.argtypes = [P, i32, i32, P]
    L.verkv_get_appended.restype = st
    L.verkv_get_row_weights.argtypes = [P, i32, i32, P, P, i32, P, P]
    L.verkv_get_row_weights.restype = st
    L.verkv_last_launch_count.argtypes = [P]
    L.verkv_last_launch_count.restype = i32
    L.verkv_set_kernel_timing.argtypes = [P, i32]
    L.verkv_set_kernel_timing.restype = st
    L.verkv_get_kernel_times.argtypes = [P, P, P, i32, P, P]
    L.verkv_get_kernel_times.restype = st
    L.verkv_status_str.argtypes = [st]
    L.verkv_status_str.restype = ctypes.c_char_p
    L.verkv_last_error.argtypes = [P]
    L.verkv_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _ptr(x):
    """Raw pointer of a torch tensor, numpy array or int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class VerKV:
    """One library context (one GPU)."""

    def __init__(self, *, n_kv_heads, n_q_heads, max_tokens, head_dim=128, n_layers=1, n_seqs=1, max_batch=1,
                 n_sink=4, n_local=128, eta=1 / 16, seed=0, sketch="int8", kv_dtype="bf16", sketch_group=128,
                 shrinkage="clipped"):
        self.cfg = Config(n_layers, n_seqs, max_batch, n_kv_heads, n_q_heads, head_dim, max_tokens, n_sink, n_local,
                          sketch_group, SHRINKAGE[shrinkage], float(eta), int(seed), SKETCH[sketch],
                          DTYPE[kv_dtype])
        self.sketch = sketch
        self.kv_dtype = kv_dtype
        h = ctypes.c_void_p()
        rc = lib().verkv_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if rc != 0:
            raise VerkvError(rc, "verkv_create failed")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().verkv_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc):
        if rc != 0:
            raise VerkvError(rc, lib().verkv_last_error(self.h).decode())

    # -- Algorithm 1
    def compress(self, layer, seq, n_tokens, kv_host, kv_dev=None, obs_q=None, W=0, tau=None, stream=None):
        stats = (HeadStats * self.cfg.n_kv_heads)()
        self._check(lib().verkv_compress(self.h, layer, seq, n_tokens, _ptr(kv_host), _ptr(kv_dev), _ptr(obs_q),
                                         int(W), _ptr(tau), _stream(stream), stats))
        return [s.as_dict() for s in stats]

    # -- Algorithm 2 + attention
    def decode(self, layer, seq_ids, q, eps, delta, out, stream=None):
        ids = np.ascontiguousarray(seq_ids, np.int32)
        self._check(lib().verkv_decode(self.h, layer, ids.ctypes.data, len(ids), _ptr(q), float(eps), float(delta),
                                       _ptr(out), _stream(stream)))

    def release(self, layer, seq):
        self._check(lib().verkv_release(self.h, layer, seq))

    def last_launch_count(self) -> int:
        return lib().verkv_last_launch_count(self.h)

    def set_kernel_timing(self, enable: bool):
        self._check(lib().verkv_set_kernel_timing(self.h, 1 if enable else 0))

    def kernel_times(self, stream=None):
        """[(kernel name, ms)] of every kernel launched by the timed calls since the last read."""
        cap = 4096
        names = (ctypes.c_char_p * cap)()
        ms = (ctypes.c_float * cap)()
        cnt = ctypes.c_int32()
        self._check(lib().verkv_get_kernel_times(self.h, names, ms, cap, ctypes.byref(cnt), _stream(stream)))
        return [(names[i].decode(), float(ms[i])) for i in range(min(cnt.value, cap))]

    # -- inspection
    def compress_state(self, layer, seq, kv_head, n, stream=None):
        c = ctypes.c_double()
        tau = np.zeros(n, np.float32)
        r = np.zeros(n, np.float32)
        flags = np.zeros(n, np.uint8)
        self._check(lib().verkv_get_compress_state(self.h, layer, seq, kv_head, ctypes.byref(c), tau.ctypes.data,
                                                   r.ctypes.data, flags.ctypes.data, _stream(stream)))
        return c.value, tau, r, flags

    def sketch_int8(self, layer, seq, kv_head, n, stream=None):
        codes = np.zeros((n, self.cfg.head_dim), np.int8)
        scale = np.zeros(n, np.float32)
        self._check(lib().verkv_get_sketch(self.h, layer, seq, kv_head, codes.ctypes.data, scale.ctypes.data, None,
                                           None, None, None, _stream(stream)))
        return codes, scale

    def sketch_2bit(self, layer, seq, kv_head, n, stream=None):
        d = self.cfg.head_dim
        ng = (n + self.cfg.sketch_group - 1) // self.cfg.sketch_group
        pairs = np.zeros(d // 8, np.int32)
        codes = np.zeros((n, d // 4), np.uint8)
        zero = np.zeros((ng, d // 4), np.uint16)
        scale = np.zeros((ng, d // 4), np.uint16)
        self._check(lib().verkv_get_sketch(self.h, layer, seq, kv_head, None, None, pairs.ctypes.data,
                                           codes.ctypes.data, zero.ctypes.data, scale.ctypes.data, _stream(stream)))
        return pairs, codes, zero, scale

    def decode_trace(self, n_rows, stream=None):
        rows = (RowTrace * n_rows)()
        self._check(lib().verkv_get_decode_trace(self.h, rows, n_rows, _stream(stream)))
        return [r.as_dict() for r in rows]

    def exact_set(self, b, h, cap, stream=None):
        out = np.zeros(max(cap, 1), np.int32)
        cnt = ctypes.c_int32()
        self._check(lib().verkv_get_exact_set(self.h, b, h, out.ctypes.data, cap, ctypes.byref(cnt), _stream(stream)))
        return out[:min(cnt.value, cap)].copy()

    def fetch_set(self, b, kv, cap, stream=None):
        out = np.zeros(max(cap, 1), np.int32)
        cnt = ctypes.c_int32()
        self._check(lib().verkv_get_fetch_set(self.h, b, kv, out.ctypes.data, cap, ctypes.byref(cnt), _stream(stream)))
        return out[:min(cnt.value, cap)].copy()

    def fetch_stats(self, b, kv, stream=None):
        """(rows the last decode needed beyond the resident ones, rows it read over the host link) of KV
        head (b, kv)."""
        nu, nh = ctypes.c_int32(), ctypes.c_int32()
        self._check(lib().verkv_get_fetch_stats(self.h, b, kv, ctypes.byref(nu), ctypes.byref(nh), _stream(stream)))
        return nu.value, nh.value

    def set_shortlist(self, k: int):
        """Appendix A.1 shortlist of k tokens per KV head scored exactly (0: off)."""
        self._check(lib().verkv_set_shortlist(self.h, int(k)))

    def shortlist(self, b, kv, cap=1024, stream=None):
        out = np.zeros(max(cap, 1), np.int32)
        cnt = ctypes.c_int32()
        self._check(lib().verkv_get_shortlist(self.h, b, kv, out.ctypes.data, cap, ctypes.byref(cnt), _stream(stream)))
        return out[:min(cnt.value, cap)].copy()

    def set_prefetch(self, rows_per_kv_head: int):
        """Rows per (sequence, KV head) the speculative prefetch may copy ahead (0 = off; default 4096)."""
        self._check(lib().verkv_set_prefetch(self.h, int(rows_per_kv_head)))

    TIMELINE_KEYS = ("decide_start", "decide_end", "prefetch_start", "prefetch_binned", "prefetch_end",
                     "attn_start", "attn_end")

    def set_timeline(self, on: bool):
        """Record the device timeline of every following decode (verkv_set_timeline)."""
        self._check(lib().verkv_set_timeline(self.h, 1 if on else 0))

    def timeline(self, stream=None):
        """Timeline of the last decode: microseconds after its scoring kernel started, per TIMELINE_KEYS
        (NaN where that kernel did not run)."""
        v = (ctypes.c_double * len(self.TIMELINE_KEYS))()
        self._check(lib().verkv_get_timeline(self.h, v, _stream(stream)))
        return dict(zip(self.TIMELINE_KEYS, list(v)))

    def prefetch_stats(self, b, kv, stream=None):
        """(rows the prefetch copied, rows the attention read from them) for KV head (b, kv), last decode."""
        nc, nu = ctypes.c_int32(), ctypes.c_int32()
        self._check(lib().verkv_get_prefetch_stats(self.h, b, kv, ctypes.byref(nc), ctypes.byref(nu), _stream(stream)))
        return nc.value, nu.value

    def set_stage_capacity(self, rows_per_kv_head: int):
        """Staging cache rows per KV head and slot (from the next compress on): STAGE_ETA_N (-2, default) =
        ceil(eta n), STAGE_ALL (-1) = all of L minus S, 0 = off, k > 0 = k rows."""
        self._check(lib().verkv_set_stage_capacity(self.h, int(rows_per_kv_head)))

    def selftest_wait_timeout(self, stream=None) -> int:
        """Run the failure-path self test; returns its status (VERKV_ETIMEOUT = 4 when the bounded wait
        gave up as intended)."""
        return int(lib().verkv_selftest_wait_timeout(self.h, _stream(stream)))

    def set_append_capacity(self, rows_per_kv_head: int):
        """Room reserved per KV head and slot for tokens appended at decode time (next compress on)."""
        self._check(lib().verkv_set_append_capacity(self.h, int(rows_per_kv_head)))

    def append(self, layer, seq, n_new, kv_new, stream=None):
        """Append n_new generated tokens to H of the slot: kv_new holds [Hkv][n_new][2][d] rows in the
        storage dtype, in device or pinned host memory."""
        self._check(lib().verkv_append(self.h, layer, seq, int(n_new), _ptr(kv_new), _stream(stream)))

    def appended(self, layer, seq) -> int:
        n = ctypes.c_int32()
        self._check(lib().verkv_get_appended(self.h, layer, seq, ctypes.byref(n)))
        return n.value

    def row_weights(self, b, h, cap, stream=None):
        w = np.zeros(max(cap, 1), np.float32)
        tok = np.zeros(max(cap, 1), np.int32)
        cnt = ctypes.c_int32()
        self._check(lib().verkv_get_row_weights(self.h, b, h, w.ctypes.data, tok.ctypes.data, cap, ctypes.byref(cnt),
                                                _stream(stream)))
        m = min(cnt.value, cap)
        return w[:m].copy(), tok[:m].copy()
