"""The C ABI: the library builds, loads without a GPU and exports every function include/verkv.h
declares; the ctypes structs match the C layouts (checked by compiling a probe against the header)."""
import ctypes
import os
import subprocess
import tempfile

import pytest

from verified_kv_cache_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def test_header_declares_the_boundary():
    names = binding.declared_functions()
    for must in ["verkv_create", "verkv_destroy", "verkv_compress", "verkv_decode", "verkv_release",
                 "verkv_get_compress_state", "verkv_get_decode_trace", "verkv_status_str", "verkv_last_error"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in binding.declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in binding.declared_functions():
        assert n in exported, n


def test_status_strings(lib):
    assert lib.verkv_status_str(0) == b"ok"
    assert lib.verkv_status_str(1) == b"invalid argument"
    assert lib.verkv_last_error(None) == b"null context"


def test_null_context_is_rejected_without_touching_the_gpu(lib):
    einval = 1
    assert lib.verkv_set_append_capacity(None, 16) == einval
    assert lib.verkv_append(None, 0, 0, 1, None, None) == einval
    assert lib.verkv_get_appended(None, 0, 0, None) == einval
    assert lib.verkv_set_stage_capacity(None, 0) == einval
    assert lib.verkv_set_shortlist(None, 8) == einval
    assert lib.verkv_selftest_wait_timeout(None, None) == einval


PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "verkv.h"
#define F(T, m) printf(#T "." #m " %zu\n", offsetof(T, m));
int main(void) {
  printf("verkv_config %zu\n", sizeof(verkv_config));
  printf("verkv_head_stats %zu\n", sizeof(verkv_head_stats));
  printf("verkv_row_trace %zu\n", sizeof(verkv_row_trace));
  F(verkv_config, eta) F(verkv_config, seed) F(verkv_config, sketch) F(verkv_config, kv_dtype)
  F(verkv_head_stats, n_resident) F(verkv_row_trace, eps_hat) F(verkv_row_trace, n_fetch)
  F(verkv_config, shrinkage) F(verkv_row_trace, n_shrunk)
  return 0;
}
"""


def test_ctypes_layouts_match_header():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        with open(src, "w") as f:
            f.write(PROBE)
        subprocess.run(["gcc", "-I", os.path.join(build.ROOT, "include"), src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.strip().splitlines())
    assert int(got["verkv_config"]) == ctypes.sizeof(binding.Config)
    assert int(got["verkv_head_stats"]) == ctypes.sizeof(binding.HeadStats)
    assert int(got["verkv_row_trace"]) == ctypes.sizeof(binding.RowTrace)
    assert int(got["verkv_config.eta"]) == binding.Config.eta.offset
    assert int(got["verkv_config.seed"]) == binding.Config.seed.offset
    assert int(got["verkv_config.sketch"]) == binding.Config.sketch.offset
    assert int(got["verkv_config.kv_dtype"]) == binding.Config.kv_dtype.offset
    assert int(got["verkv_head_stats.n_resident"]) == binding.HeadStats.n_resident.offset
    assert int(got["verkv_row_trace.eps_hat"]) == binding.RowTrace.eps_hat.offset
    assert int(got["verkv_row_trace.n_fetch"]) == binding.RowTrace.n_fetch.offset
    assert int(got["verkv_config.shrinkage"]) == binding.Config.shrinkage.offset
    assert int(got["verkv_row_trace.n_shrunk"]) == binding.RowTrace.n_shrunk.offset


def test_create_rejects_bad_configs_without_touching_the_gpu(lib):
    # argument checks run before any CUDA call
    cfg = binding.Config(1, 1, 1, 8, 30, 128, 1024, 4, 64, 128, 0, 0.125, 0, 1, 0)  # 30 % 8 != 0
    h = ctypes.c_void_p()
    assert lib.verkv_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
    cfg = binding.Config(1, 1, 1, 8, 32, 64, 1024, 4, 64, 128, 0, 0.125, 0, 1, 0)   # head_dim 64
    assert lib.verkv_create(ctypes.byref(cfg), ctypes.byref(h)) == 5
    cfg = binding.Config(1, 1, 1, 8, 32, 128, 1024, 4, 64, 128, 0, 1.5, 0, 1, 0)    # eta > 1
    assert lib.verkv_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
    cfg = binding.Config(1, 1, 1, 8, 32, 128, 1024, 4, 64, 128, 2, 0.125, 0, 1, 0)  # unknown shrinkage
    assert lib.verkv_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
