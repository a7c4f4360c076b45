"""Host-side checks of the C-ABI library that need no GPU.

The library builds for sm_103a on this machine, loads, exports every entry
point include/rlk.h declares, and its host logic (tile tree, workspace
sizes, argument validation) behaves as documented.  No call here reaches a
kernel launch: every call either is host-only or is refused by argument
validation before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest

from invariant_selected_token_gb300 import binding, build
from oracle import linear_logprob as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# the largest row count any call takes, as include/rlk.h defines it
MAX_ROWS = int(re.search(r"#define RLK_MAX_ROWS (\d+)",
                         open(os.path.join(ROOT, "include", "rlk.h")).read()).group(1))


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "rlk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rlk_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    syms = declared_symbols()
    assert len(syms) >= 11
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [s for s in syms if s not in exported]
    assert not missing, missing
    for s in syms:
        getattr(L, s)  # resolvable through ctypes as well
    assert sorted(binding.EXPORTED) == syms


def test_contract_id_and_fingerprint(L):
    assert binding.contract_id() == "rlk-linlogp-v1"
    fp = binding.build_fingerprint()
    assert "rlk-linlogp-v1" in fp and "sm_103a" in fp and "-fmad=false" in fp
    assert L.rlk_status_string(6) == b"RLK_ERR_TARGET_RANGE"


@pytest.mark.parametrize("V", [1, 2, 129, 1000, 1024, 131072, 151936, 262144])
@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_shard_ranges_match_oracle_tree(L, V, n):
    nt = (V + 127) // 128
    if n > nt:
        with pytest.raises(binding.RlkError) as e:
            binding.shard_range(V, n, 0)
        assert e.value.code == 2
        return
    assert binding.shard_ranges(V, n) == O.shard_vocab_ranges(V, n)


def test_shard_range_errors(L):
    for args, code in [((0, 1, 0), 1), ((1000, 3, 0), 2), ((1000, 16, 0), 2), ((262145, 1, 0), 2),
                       ((1000, 4, 4), 1), ((1000, 4, -1), 1)]:
        with pytest.raises(binding.RlkError) as e:
            binding.shard_range(*args)
        assert e.value.code == code, args


def test_workspace_size(L):
    T, V = 4096, 151936
    nt = 1187
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert binding.workspace_size(T, V, 4) == a(T * nt * 8) + a(T * 4) + a(T * 4 * 16)
    assert L.rlk_workspace_size(10, 1000, 3) == 0
    assert L.rlk_workspace_size(-1, 1000, 1) == 0
    assert L.rlk_workspace_size(0, 1000, 1) == 0


def _call_full(L, hidden=0x10000, W=0x20000, targets=0x30000, active=None, T=4, H=64, V=1000,
               n_shards=1, lp=0x40000, lse=0x50000, ws=0x60000, ws_bytes=1 << 20, status=None):
    return L.rlk_linear_logprob(hidden, W, targets, active, T, H, V, n_shards, lp, lse, ws,
                                ws_bytes, status, None)


def test_argument_validation_refuses_before_any_cuda_call(L):
    # every case below is refused by host checks; the pointers are never dereferenced
    assert _call_full(L, hidden=None) == 1
    assert _call_full(L, lp=None) == 1
    assert _call_full(L, T=-1) == 1
    assert _call_full(L, H=96) == 2
    assert _call_full(L, H=0) == 2
    assert _call_full(L, H=(1 << 20) + 64) == 2  # beyond the widest hidden size served
    assert _call_full(L, V=262145) == 2
    assert _call_full(L, V=0) == 1
    assert _call_full(L, n_shards=3) == 2
    assert _call_full(L, V=300, n_shards=4) == 2      # 3 tiles cannot hold 4 shards
    assert _call_full(L, hidden=0x10008) == 3
    assert _call_full(L, W=0x20004) == 3
    assert _call_full(L, ws=0x60010) == 3
    assert _call_full(L, ws_bytes=100) == 4
    assert _call_full(L, ws=None) == 1
    assert _call_full(L, T=0) == 0                    # empty batch: no-op
    assert _call_full(L, T=MAX_ROWS + 1) == 1         # beyond the largest row count
    assert L.rlk_workspace_size(MAX_ROWS + 1, 1000, 1) == 0
    # shard variant and merge
    assert L.rlk_linear_logprob_shard(0x10000, 0x20000, 0x30000, None, 4, 64, 1000, 4, 4, 0x40000,
                                      0x60000, 1 << 20, None, None) == 1
    assert L.rlk_linear_logprob_shard(0x10000, 0x20000, 0x30000, None, 4, 64, 1000, 4, 1, 0x40008,
                                      0x60000, 1 << 20, None, None) == 3
    arr = (ctypes.c_void_p * 2)(0x1000, None)
    assert L.rlk_lse_merge(ctypes.cast(arr, ctypes.c_void_p), 2, 4, None, 0x40000, 0x50000, None,
                           None) == 1
    assert L.rlk_lse_merge(ctypes.cast(arr, ctypes.c_void_p), 3, 4, None, 0x40000, 0x50000, None,
                           None) == 2
    assert L.rlk_debug_logits(0x10000, 0x20000, 4, 100, 10, 0x40000, None, None) == 2


def test_materialised_logits_validation(L):
    f = L.rlk_logits_logprob
    ok = dict(logits=0x10000, dtype=0, ld=1024, targets=0x30000, T=4, V=1000, n=1, lp=0x40000,
              lse=0x50000, ws=0x60000, wsb=1 << 20)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["logits"], a["dtype"], a["ld"], a["targets"], None, a["T"], a["V"], a["n"],
                 a["lp"], a["lse"], a["ws"], a["wsb"], None, None)
    assert call(dtype=2) == 2
    assert call(ld=999) == 1          # ld < V
    assert call(logits=0x10002) == 3  # fp32 elements need 4-byte alignment
    assert call(dtype=1, logits=0x10001) == 3  # bf16 elements need 2-byte alignment
    assert call(V=0) == 1
    assert call(n=3) == 2
    assert call(targets=None) == 1
    assert call(wsb=10) == 4
    assert call(T=0) == 0
    assert call(T=MAX_ROWS + 1) == 1
    g = L.rlk_log_softmax
    assert g(0x10000, 0, 1024, None, 4, 1000, None, 0x50000, 0x60000, 1 << 20, None, None) == 1
    assert g(0x10001, 0, 1001, None, 4, 1000, 0x40000, 0x50000, 0x60000, 1 << 20, None, None) == 3


def test_training_pair_validation(L):
    # the saving forward and the backward from saved logits: host checks only
    f = L.rlk_linear_logprob_save_logits
    ok = dict(h=0x10000, W=0x20000, tg=0x30000, T=4, H=64, V=1000, n=1, lp=0x40000, lse=0x50000,
              lg=0x70000, ld=1000, ws=0x60000, wsb=1 << 20)

    def fwd(**kw):
        a = dict(ok, **kw)
        return f(a["h"], a["W"], a["tg"], None, a["T"], a["H"], a["V"], a["n"], a["lp"], a["lse"],
                 a["lg"], a["ld"], a["ws"], a["wsb"], None, None)
    assert fwd(lg=None) == 1
    assert fwd(ld=996) == 1           # ld < V
    assert fwd(ld=1002) == 3          # rows must start on 16-byte boundaries
    assert fwd(lg=0x70008) == 3
    assert fwd(n=3) == 2
    assert fwd(wsb=10) == 4
    assert fwd(T=0) == 0
    b = L.rlk_linear_logprob_backward_from_logits
    okb = dict(lg=0x70000, ld=1000, h=0x10000, W=0x20000, tg=0x30000, g=0x40000, lse=0x50000, T=4,
               H=64, V=1000, dh=0x80000, dW=0x90000, ws=0x60000, wsb=1 << 30)

    def bwd(**kw):
        a = dict(okb, **kw)
        return b(a["lg"], a["ld"], a["h"], a["W"], a["tg"], None, a["g"], a["lse"], a["T"], a["H"],
                 a["V"], a["dh"], a["dW"], a["ws"], a["wsb"], None, None)
    assert bwd(lg=None) == 1
    assert bwd(ld=999) == 1
    assert bwd(ld=1001) == 3
    assert bwd(lg=0x70004) == 3
    assert bwd(dh=None, dW=None) == 1
    assert bwd(wsb=10) == 4
    assert bwd(T=0) == 0


def test_rmsnorm_validation(L):
    f = L.rlk_rmsnorm
    import ctypes as C
    ok = (0x10000, None, 0x20000, C.c_float(1e-6), 4, 4096, 0x30000, None, None)
    assert f(*ok[:4], 4, 100, *ok[6:]) == 2           # H % 64
    assert f(*ok[:4], 4, 16384, *ok[6:]) == 2         # H > 8192
    assert f(0x10000, None, 0x20000, C.c_float(0.0), 4, 4096, 0x30000, None, None) == 1
    assert f(0x10000, None, 0x20000, C.c_float(1e-6), 4, 4096, 0x30000, 0x40000, None) == 1
    assert f(0x10008, None, 0x20000, C.c_float(1e-6), 4, 4096, 0x30000, None, None) == 3
    assert f(0x10000, None, 0x20000, C.c_float(1e-6), 0, 4096, 0x30000, None, None) == 0
    assert f(0x10000, None, 0x20000, C.c_float(1e-6), MAX_ROWS + 1, 4096, 0x30000, None,
             None) == 1
