"""Python binding of librlk.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this
module checks tensor dtypes/devices/contiguity, allocates outputs and the
workspace through torch (device memory and streams are torch's), and passes
raw pointers to the C-ABI calls declared in include/rlk.h.  If librlk.so is
missing, every call raises -- there is no other implementation to fall back
to.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librlk.so")

STATUS_NAMES = {0: "RLK_OK", 1: "RLK_ERR_INVALID_ARG", 2: "RLK_ERR_UNSUPPORTED",
                3: "RLK_ERR_ALIGNMENT", 4: "RLK_ERR_WORKSPACE", 5: "RLK_ERR_CUDA",
                6: "RLK_ERR_TARGET_RANGE", 7: "RLK_ERR_TIMEOUT"}
RLK_ERR_INVALID_ARG = 1
RLK_ERR_ALIGNMENT = 3
RLK_ERR_TARGET_RANGE = 6
RLK_ERR_TIMEOUT = 7
VOCAB_TILE = 128

EXPORTED = ["rlk_contract_id", "rlk_build_fingerprint", "rlk_status_string", "rlk_shard_range",
            "rlk_workspace_size", "rlk_linear_logprob", "rlk_linear_logprob_shard",
            "rlk_lse_merge", "rlk_tile_partials", "rlk_tile_merge", "rlk_debug_logits",
            "rlk_linear_logprob_static_ws", "rlk_logits_logprob", "rlk_log_softmax",
            "rlk_backward_workspace_size", "rlk_linear_logprob_backward", "rlk_rmsnorm",
            "rlk_debug_primitive_hash", "rlk_linear_logprob_save_logits",
            "rlk_linear_logprob_backward_from_logits"]
DTYPES = {torch.float32: 0, torch.bfloat16: 1}


class RlkError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__("%s returned %s" % (where, STATUS_NAMES.get(code, str(code))))
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("librlk.so not found at %s; build it with "
                               "`python -m invariant_selected_token_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        L.rlk_contract_id.restype = ctypes.c_char_p
        L.rlk_contract_id.argtypes = []
        L.rlk_build_fingerprint.restype = ctypes.c_char_p
        L.rlk_build_fingerprint.argtypes = []
        L.rlk_status_string.restype = ctypes.c_char_p
        L.rlk_status_string.argtypes = [i32]
        L.rlk_shard_range.restype = i32
        L.rlk_shard_range.argtypes = [i64, i32, i32, P, P]
        L.rlk_workspace_size.restype = sz
        L.rlk_workspace_size.argtypes = [i64, i64, i32]
        L.rlk_linear_logprob.restype = i32
        L.rlk_linear_logprob.argtypes = [P, P, P, P, i64, i64, i64, i32, P, P, P, sz, P, P]
        L.rlk_linear_logprob_shard.restype = i32
        L.rlk_linear_logprob_shard.argtypes = [P, P, P, P, i64, i64, i64, i32, i32, P, P, sz, P, P]
        L.rlk_lse_merge.restype = i32
        L.rlk_lse_merge.argtypes = [P, i32, i64, P, P, P, P, P]
        L.rlk_tile_partials.restype = i32
        L.rlk_tile_partials.argtypes = [P, P, P, P, i64, i64, i64, i32, P, sz, P, P]
        L.rlk_tile_merge.restype = i32
        L.rlk_tile_merge.argtypes = [P, P, i64, i64, i32, P, P, P, sz, P, P]
        L.rlk_debug_logits.restype = i32
        L.rlk_debug_logits.argtypes = [P, P, i64, i64, i64, P, P, P]
        L.rlk_logits_logprob.restype = i32
        L.rlk_logits_logprob.argtypes = [P, i32, i64, P, P, i64, i64, i32, P, P, P, sz, P, P]
        L.rlk_backward_workspace_size.restype = sz
        L.rlk_backward_workspace_size.argtypes = [i64, i64, i64]
        L.rlk_linear_logprob_backward.restype = i32
        L.rlk_linear_logprob_backward.argtypes = [P, P, P, P, P, P, i64, i64, i64, P, P, P, sz, P,
                                                  P]
        L.rlk_linear_logprob_save_logits.restype = i32
        L.rlk_linear_logprob_save_logits.argtypes = [P, P, P, P, i64, i64, i64, i32, P, P, P, i64,
                                                     P, sz, P, P]
        L.rlk_linear_logprob_backward_from_logits.restype = i32
        L.rlk_linear_logprob_backward_from_logits.argtypes = [P, i64, P, P, P, P, P, P, i64, i64,
                                                              i64, P, P, P, sz, P, P]
        L.rlk_rmsnorm.restype = i32
        L.rlk_rmsnorm.argtypes = [P, P, P, ctypes.c_float, i64, i64, P, P, P]
        L.rlk_log_softmax.restype = i32
        L.rlk_log_softmax.argtypes = [P, i32, i64, P, i64, i64, P, P, P, sz, P, P]
        L.rlk_debug_primitive_hash.restype = i32
        L.rlk_debug_primitive_hash.argtypes = [i32, ctypes.c_uint32, ctypes.c_uint64, P, P]
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise RlkError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on(device):
    """Make the tensors' device current for the call: the library launches on the calling
    thread's current device."""
    return torch.cuda.device(device)


def _stream(device: torch.device, stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _require(t: torch.Tensor, dtype, name: str, device=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be on a CUDA device" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))


# ----------------------------------------------------------------- host-only calls
def contract_id() -> str:
    return lib().rlk_contract_id().decode()


def build_fingerprint() -> str:
    return lib().rlk_build_fingerprint().decode()


def shard_range(V: int, n_shards: int, shard: int) -> Tuple[int, int]:
    b, e = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().rlk_shard_range(V, n_shards, shard, ctypes.byref(b), ctypes.byref(e)),
           "rlk_shard_range")
    return b.value, e.value


def workspace_size(T: int, V: int, n_shards: int = 1) -> int:
    n = lib().rlk_workspace_size(T, V, n_shards)
    if n == 0 and T > 0:
        raise RlkError(1, "rlk_workspace_size")
    return int(n)


def new_workspace(T: int, V: int, n_shards: int, device) -> torch.Tensor:
    return torch.empty(max(256, workspace_size(T, V, n_shards)), dtype=torch.uint8, device=device)


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def raise_on_device_status(status: torch.Tensor):
    """Synchronise on the status word and raise for the first error bit set."""
    word = int(status.item())
    for code in sorted(STATUS_NAMES):
        if code and word & (1 << code):
            raise RlkError(code, "device status 0x%x" % word)


# ----------------------------------------------------------------- device calls
def linear_logprob(hidden: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                   active: Optional[torch.Tensor] = None, n_shards: int = 1,
                   out_logprob: Optional[torch.Tensor] = None,
                   out_lse: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None
                   ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(logprob [T], lse [T]) fp32 for bf16 hidden [T,H], W [V,H], int32 targets [T]."""
    dev = hidden.device
    _require(hidden, torch.bfloat16, "hidden", ndim=2)
    _require(W, torch.bfloat16, "W", dev, ndim=2)
    _require(targets, torch.int32, "targets", dev, ndim=1)
    if active is not None:
        _require(active, torch.uint8, "active", dev, ndim=1)
    T, H = hidden.shape
    V = W.shape[0]
    if W.shape[1] != H or targets.shape[0] != T or (active is not None and active.shape[0] != T):
        raise ValueError("shape mismatch")
    if out_logprob is None:
        out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, V, n_shards, dev)
    with _on(dev):
        _check(lib().rlk_linear_logprob(_ptr(hidden), _ptr(W), _ptr(targets), _ptr(active), T, H, V,
                                        n_shards, _ptr(out_logprob), _ptr(out_lse), _ptr(workspace),
                                        workspace.numel(), _ptr(status), _stream(dev, stream)),
               "rlk_linear_logprob")
    return out_logprob, out_lse


def tile_partials(hidden, W, targets, active, n_shards, workspace, status=None, stream=None):
    dev = hidden.device
    T, H = hidden.shape
    with _on(dev):
        _check(lib().rlk_tile_partials(_ptr(hidden), _ptr(W), _ptr(targets), _ptr(active), T, H,
                                       W.shape[0], n_shards, _ptr(workspace), workspace.numel(),
                                       _ptr(status), _stream(dev, stream)), "rlk_tile_partials")


def tile_merge(targets, active, V, n_shards, out_logprob, out_lse, workspace, status=None,
               stream=None):
    dev = targets.device
    T = targets.shape[0]
    with _on(dev):
        _check(lib().rlk_tile_merge(_ptr(targets), _ptr(active), T, V, n_shards, _ptr(out_logprob),
                                    _ptr(out_lse), _ptr(workspace), workspace.numel(), _ptr(status),
                                    _stream(dev, stream)), "rlk_tile_merge")


def workspace_records(workspace: torch.Tensor, T: int, V: int, n_shards: int) -> torch.Tensor:
    """View of the shard records rlk_linear_logprob leaves in its workspace: int32 [n_shards, T, 4]."""
    nt = (V + VOCAB_TILE - 1) // VOCAB_TILE
    a256 = lambda x: (x + 255) & ~255  # noqa: E731
    off = a256(T * nt * 8) + a256(T * 4)
    return workspace[off:off + n_shards * T * 16].view(torch.int32).view(n_shards, T, 4)


def linear_logprob_shard(hidden, W_shard, targets, active, V_total: int, n_shards: int,
                         shard: int, out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, status=None, stream=None
                         ) -> torch.Tensor:
    """One shard's records as int32 [T, 4] (m, s, tgt as fp32 bits; owned as uint32)."""
    dev = hidden.device
    _require(hidden, torch.bfloat16, "hidden", ndim=2)
    _require(W_shard, torch.bfloat16, "W_shard", dev, ndim=2)
    _require(targets, torch.int32, "targets", dev, ndim=1)
    T, H = hidden.shape
    vb, ve = shard_range(V_total, n_shards, shard)
    if W_shard.shape[0] != ve - vb:
        raise ValueError("W_shard has %d rows, shard %d covers %d" % (W_shard.shape[0], shard, ve - vb))
    if out is None:
        out = torch.empty((T, 4), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, ve - vb, 1, dev)
    with _on(dev):
        _check(lib().rlk_linear_logprob_shard(_ptr(hidden), _ptr(W_shard), _ptr(targets),
                                              _ptr(active), T, H, V_total, n_shards, shard,
                                              _ptr(out),
                                              _ptr(workspace), workspace.numel(), _ptr(status),
                                              _stream(dev, stream)), "rlk_linear_logprob_shard")
    return out


def lse_merge(partials: Sequence[torch.Tensor], active=None, out_logprob=None, out_lse=None,
              status=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    n = len(partials)
    dev = partials[0].device
    T = partials[0].shape[0]
    for p in partials:
        _require(p, torch.int32, "partial", dev, ndim=2)
    arr = (ctypes.c_void_p * n)(*[p.data_ptr() for p in partials])
    if out_logprob is None:
        out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    with _on(dev):
        _check(lib().rlk_lse_merge(ctypes.cast(arr, ctypes.c_void_p), n, T, _ptr(active),
                                   _ptr(out_logprob), _ptr(out_lse), _ptr(status),
                                   _stream(dev, stream)), "rlk_lse_merge")
    return out_logprob, out_lse


def debug_logits(hidden: torch.Tensor, W: torch.Tensor, status=None, stream=None) -> torch.Tensor:
    dev = hidden.device
    _require(hidden, torch.bfloat16, "hidden", ndim=2)
    _require(W, torch.bfloat16, "W", dev, ndim=2)
    T, H = hidden.shape
    V = W.shape[0]
    out = torch.empty((T, V), dtype=torch.float32, device=dev)
    with _on(dev):
        _check(lib().rlk_debug_logits(_ptr(hidden), _ptr(W), T, H, V, _ptr(out), _ptr(status),
                                      _stream(dev, stream)), "rlk_debug_logits")
    return out


def shard_ranges(V: int, n_shards: int) -> List[Tuple[int, int]]:
    return [shard_range(V, n_shards, r) for r in range(n_shards)]


def _logits_view(logits: torch.Tensor, V: Optional[int]):
    if logits.dtype not in DTYPES:
        raise TypeError("logits must be float32 or bfloat16")
    if not logits.is_cuda or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D CUDA tensor with unit column stride")
    T = logits.shape[0]
    V = logits.shape[1] if V is None else V
    return T, V, logits.stride(0) if T > 1 else V


def logits_logprob(logits: torch.Tensor, targets: torch.Tensor, active=None, n_shards: int = 1,
                   out_logprob=None, out_lse=None, workspace=None, status=None, stream=None
                   ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(logprob, lse) of materialised fp32/bf16 logits [T, V] (rows may be padded)."""
    dev = logits.device
    T, V, ld = _logits_view(logits, None)
    _require(targets, torch.int32, "targets", dev, ndim=1)
    if out_logprob is None:
        out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, V, n_shards, dev)
    with _on(dev):
        _check(lib().rlk_logits_logprob(_ptr(logits), DTYPES[logits.dtype], ld, _ptr(targets),
                                        _ptr(active), T, V, n_shards, _ptr(out_logprob),
                                        _ptr(out_lse),
                                        _ptr(workspace), workspace.numel(), _ptr(status),
                                        _stream(dev, stream)), "rlk_logits_logprob")
    return out_logprob, out_lse


def log_softmax(logits: torch.Tensor, active=None, out=None, out_lse=None, workspace=None,
                status=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """(log_softmax [T, V] fp32, lse [T]) of materialised fp32/bf16 logits."""
    dev = logits.device
    T, V, ld = _logits_view(logits, None)
    if out is None:
        out = torch.empty((T, V), dtype=torch.float32, device=dev)
    if out_lse is None:
        out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, V, 1, dev)
    with _on(dev):
        _check(lib().rlk_log_softmax(_ptr(logits), DTYPES[logits.dtype], ld, _ptr(active), T, V,
                                     _ptr(out), _ptr(out_lse), _ptr(workspace), workspace.numel(),
                                     _ptr(status), _stream(dev, stream)), "rlk_log_softmax")
    return out, out_lse


def backward_workspace_size(T: int, H: int, V: int) -> int:
    return int(lib().rlk_backward_workspace_size(T, H, V))


def backward_grad_view(workspace: torch.Tensor, T: int, V: int) -> torch.Tensor:
    """The bf16 logit gradient G [T, V] the backward leaves at the start of its workspace."""
    ld = (V + 7) // 8 * 8
    return workspace[:T * ld * 2].view(torch.bfloat16).view(T, ld)[:, :V]


def linear_logprob_backward(hidden, W, targets, grad_logprob, lse, active=None,
                            want_hidden: bool = True, want_W: bool = True, grad_hidden=None,
                            grad_W=None, workspace=None, status=None, stream=None):
    """(grad_hidden [T,H] or None, grad_W [V,H] or None) of sum_t g[t] * logprob[t]."""
    dev = hidden.device
    _require(hidden, torch.bfloat16, "hidden", ndim=2)
    _require(W, torch.bfloat16, "W", dev, ndim=2)
    _require(targets, torch.int32, "targets", dev, ndim=1)
    _require(grad_logprob, torch.float32, "grad_logprob", dev, ndim=1)
    _require(lse, torch.float32, "lse", dev, ndim=1)
    T, H = hidden.shape
    V = W.shape[0]
    if want_hidden and grad_hidden is None:
        grad_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
    if want_W and grad_W is None:
        grad_W = torch.empty((V, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(256, backward_workspace_size(T, H, V)), dtype=torch.uint8,
                                device=dev)
    with _on(dev):
        _check(lib().rlk_linear_logprob_backward(
            _ptr(hidden), _ptr(W), _ptr(targets), _ptr(active), _ptr(grad_logprob), _ptr(lse),
            T, H, V,
            _ptr(grad_hidden if want_hidden else None), _ptr(grad_W if want_W else None),
            _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev, stream)),
            "rlk_linear_logprob_backward")
    return (grad_hidden if want_hidden else None), (grad_W if want_W else None)


def linear_logprob_save_logits(hidden, W, targets, active=None, n_shards: int = 1, logits=None,
                               workspace=None, status=None, stream=None):
    """(logprob [T], lse [T], logits fp32 [T, ld]): rlk_linear_logprob's outputs and bits,
    plus every row's fp32 logits for rlk_linear_logprob_backward_from_logits.  `logits`, if
    given, is a float32 [T, ld] tensor with ld >= V a multiple of 4 (its first V columns are
    written)."""
    dev = hidden.device
    _require(hidden, torch.bfloat16, "hidden", ndim=2)
    _require(W, torch.bfloat16, "W", dev, ndim=2)
    _require(targets, torch.int32, "targets", dev, ndim=1)
    if active is not None:
        _require(active, torch.uint8, "active", dev, ndim=1)
    T, H = hidden.shape
    V = W.shape[0]
    if W.shape[1] != H or targets.shape[0] != T or (active is not None and active.shape[0] != T):
        raise ValueError("shape mismatch")
    if logits is None:
        logits = torch.empty((T, (V + 3) // 4 * 4), dtype=torch.float32, device=dev)
    _require(logits, torch.float32, "logits", dev, ndim=2)
    if logits.stride(1) != 1 or logits.shape[0] != T:
        raise ValueError("logits must be [T, ld] with unit column stride")
    out_logprob = torch.empty(T, dtype=torch.float32, device=dev)
    out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(T, V, n_shards, dev)
    with _on(dev):
        _check(lib().rlk_linear_logprob_save_logits(
            _ptr(hidden), _ptr(W), _ptr(targets), _ptr(active), T, H, V, n_shards,
            _ptr(out_logprob), _ptr(out_lse), _ptr(logits), logits.stride(0), _ptr(workspace),
            workspace.numel(), _ptr(status), _stream(dev, stream)),
            "rlk_linear_logprob_save_logits")
    return out_logprob, out_lse, logits


def linear_logprob_backward_from_logits(logits, hidden, W, targets, grad_logprob, lse,
                                        active=None, want_hidden: bool = True,
                                        want_W: bool = True, grad_hidden=None, grad_W=None,
                                        workspace=None, status=None, stream=None):
    """linear_logprob_backward with G formed from the saved fp32 logits [T, ld] of
    linear_logprob_save_logits (same bits)."""
    dev = hidden.device
    _require(logits, torch.float32, "logits", dev, ndim=2)
    _require(hidden, torch.bfloat16, "hidden", ndim=2)
    _require(W, torch.bfloat16, "W", dev, ndim=2)
    _require(targets, torch.int32, "targets", dev, ndim=1)
    _require(grad_logprob, torch.float32, "grad_logprob", dev, ndim=1)
    _require(lse, torch.float32, "lse", dev, ndim=1)
    T, H = hidden.shape
    V = W.shape[0]
    if logits.stride(1) != 1 or logits.shape[0] != T:
        raise ValueError("logits must be [T, ld] with unit column stride")
    if want_hidden and grad_hidden is None:
        grad_hidden = torch.empty((T, H), dtype=torch.float32, device=dev)
    if want_W and grad_W is None:
        grad_W = torch.empty((V, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(256, backward_workspace_size(T, H, V)), dtype=torch.uint8,
                                device=dev)
    with _on(dev):
        _check(lib().rlk_linear_logprob_backward_from_logits(
            _ptr(logits), logits.stride(0), _ptr(hidden), _ptr(W), _ptr(targets), _ptr(active),
            _ptr(grad_logprob), _ptr(lse), T, H, V,
            _ptr(grad_hidden if want_hidden else None), _ptr(grad_W if want_W else None),
            _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev, stream)),
            "rlk_linear_logprob_backward_from_logits")
    return (grad_hidden if want_hidden else None), (grad_W if want_W else None)


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
            residual: Optional[torch.Tensor] = None, want_residual_out: bool = False,
            out=None, residual_out=None, stream=None):
    """Strict RMSNorm -> (out bf16 [T, H], residual_out bf16 [T, H] or None)."""
    dev = x.device
    _require(x, torch.bfloat16, "x", ndim=2)
    _require(gamma, torch.bfloat16, "gamma", dev, ndim=1)
    if residual is not None:
        _require(residual, torch.bfloat16, "residual", dev, ndim=2)
    T, H = x.shape
    if out is None:
        out = torch.empty_like(x)
    if want_residual_out and residual_out is None:
        residual_out = torch.empty_like(x)
    with _on(dev):
        _check(lib().rlk_rmsnorm(_ptr(x), _ptr(residual), _ptr(gamma), float(eps), T, H, _ptr(out),
                                 _ptr(residual_out if want_residual_out else None),
                                 _stream(dev, stream)), "rlk_rmsnorm")
    return out, (residual_out if want_residual_out else None)


PRIMITIVES = {"exp": 0, "exp_x2": 1, "log": 2, "rsqrt": 3}


def primitive_hash(which: str, first: int, count: int, device, stream=None) -> int:
    """Position-weighted 64-bit sum of one contract primitive over fp32 bit patterns
    [first, first + count), evaluated on the device (see rlk_debug_primitive_hash)."""
    out = torch.zeros(1, dtype=torch.int64, device=device)
    with _on(torch.device(device)):
        _check(lib().rlk_debug_primitive_hash(PRIMITIVES[which], first, count, _ptr(out),
                                              _stream(torch.device(device), stream)),
               "rlk_debug_primitive_hash")
    return int(out.item()) & ((1 << 64) - 1)
