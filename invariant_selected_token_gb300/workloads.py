"""Seeded synthetic inputs for the selected-token logprob.

This module only *makes inputs*: bf16 hidden states, a bf16 output-head
weight matrix, int32 target ids and a uint8 activity mask.  It holds none of
the logprob arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method's code.

Shapes and distributions follow the workloads the vLLM RL-Kernel pages
describe ("vLLM RL-Kernel v0.1.0", section "AMD Instinct MI300X での検証結果";
the Hungarian report's experiment paragraph: Qwen3-8B, BF16, seed 1234,
8 samples per prompt, responses of at most 6912 tokens):

* ``tiny``          T=64, H=256, V=1024, hidden ~N(0,1), W ~N(0,1/H), uniform targets.
* ``packed``        T=4096 (8 x 512), H=4096, V=151936, RMS-normalised hidden rows,
                    W ~N(0, 0.02), 90 % of targets drawn among the row's top-10
                    logits and 10 % uniform.
* ``decode_rows``   T in {1, 8, 64, 256} rows drawn from ``packed``.
* ``grpo_long``     8 prompts x 8 samples, prompt length U[64,512] (inactive),
                    response length U[256,6912] (active), packed into 8192-row chunks.
* ``sweep_set``     a fixed 8192-token set with the ``packed`` distributions.
* ``exact_case``    small-integer grids whose logits are exact in fp32 in any
                    summation order (used for bit-level pins).

bf16 values travel as ``uint16`` bit patterns in numpy (numpy has no bf16)
and as ``torch.bfloat16`` on the device.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

H_QWEN3_8B = 4096
V_QWEN3_8B = 151936


# --------------------------------------------------------------------------
# bf16 encoding (round to nearest even), numpy side
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    """One batch of inputs.  numpy arrays; ``hidden``/``W`` are bf16 bits."""
    name: str
    hidden: np.ndarray          # uint16 [T, H]
    W: np.ndarray               # uint16 [V, H]
    targets: np.ndarray         # int32 [T]
    active: Optional[np.ndarray] = None   # uint8 [T] or None (all active)
    n_shards: int = 1
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.hidden.shape[0])

    @property
    def H(self) -> int:
        return int(self.hidden.shape[1])

    @property
    def V(self) -> int:
        return int(self.W.shape[0])


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# Independent device-generator streams per purpose: the weights, the hidden
# rows and the target draws of one seed must not come from the same stream
# (identical streams would make hidden row t a rescaled copy of W row t).
_PURPOSE = {"weights": 1, "hidden": 2, "targets": 3}


def _stream_seed(seed: int, purpose: str) -> int:
    return (seed * 0x9E3779B1 + _PURPOSE[purpose] * 0x85EBCA77) % (1 << 62)


# --------------------------------------------------------------------------
# small numpy workloads (CPU tests and GPU parity at oracle-friendly sizes)
# --------------------------------------------------------------------------
def tiny(seed: int = 0) -> Workload:
    """T=64, H=256, V=1024, 2 shards; hidden N(0,1), W N(0,1/H), uniform targets."""
    return small_case(64, 256, 1024, seed=seed, n_shards=2, name="tiny")


def small_case(T: int, H: int, V: int, seed: int, n_shards: int = 1,
               w_std: Optional[float] = None, inactive_frac: float = 0.0,
               name: str = "small") -> Workload:
    """Gaussian hidden rows and head weights at a chosen size (ragged sizes allowed)."""
    rng = _rng(seed)
    hidden = rng.standard_normal((T, H), dtype=np.float32)
    std = (1.0 / np.sqrt(H)) if w_std is None else w_std
    W = (rng.standard_normal((V, H), dtype=np.float32) * np.float32(std)).astype(np.float32)
    targets = rng.integers(0, V, size=T, dtype=np.int64).astype(np.int32)
    active = None
    if inactive_frac > 0.0:
        active = (rng.random(T) >= inactive_frac).astype(np.uint8)
    return Workload(name, f32_to_bf16_bits(hidden), f32_to_bf16_bits(W), targets,
                    active, n_shards, {"seed": seed})


def exact_case(T: int, H: int, V: int, seed: int, n_shards: int = 1,
               h_levels: int = 8, w_levels: int = 4, inactive_frac: float = 0.0,
               name: str = "exact") -> Workload:
    """Inputs on a coarse grid: hidden = k/8 (|k| <= h_levels), W = j/64 (|j| <= w_levels).

    Every product is a multiple of 2**-9 and every partial sum an integer
    multiple of 2**-9 below 2**(24-9) in magnitude (for H * h_levels * w_levels
    < 2**24), so each logit is exactly representable in fp32 whatever the
    summation order.  That makes the fp32 logits known exactly on the CPU.
    """
    assert H * h_levels * w_levels < (1 << 24)
    rng = _rng(seed)
    k = rng.integers(-h_levels, h_levels + 1, size=(T, H)).astype(np.float32) / np.float32(8.0)
    j = rng.integers(-w_levels, w_levels + 1, size=(V, H)).astype(np.float32) / np.float32(64.0)
    targets = rng.integers(0, V, size=T, dtype=np.int64).astype(np.int32)
    active = None
    if inactive_frac > 0.0:
        active = (rng.random(T) >= inactive_frac).astype(np.uint8)
    hb, wb = f32_to_bf16_bits(k), f32_to_bf16_bits(j)
    assert np.array_equal(bf16_bits_to_f32(hb), k) and np.array_equal(bf16_bits_to_f32(wb), j)
    return Workload(name, hb, wb, targets, active, n_shards, {"seed": seed, "exact": True})


# --------------------------------------------------------------------------
# Qwen3-8B-shaped workloads, generated on the device with torch
# --------------------------------------------------------------------------
def _torch():
    import torch  # noqa: WPS433 (imported lazily: CPU-only users never need it)
    return torch


def head_weights(device, seed: int = 1234, V: int = V_QWEN3_8B, H: int = H_QWEN3_8B,
                 std: float = 0.02):
    """W ~ N(0, std) as bf16 [V, H] on ``device`` (seeded torch generator)."""
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(_stream_seed(seed, "weights"))
    W = torch.empty((V, H), dtype=torch.bfloat16, device=device)
    rows = 8192
    for r0 in range(0, V, rows):
        r1 = min(V, r0 + rows)
        W[r0:r1] = (torch.randn((r1 - r0, H), generator=g, device=device,
                                dtype=torch.float32) * std).to(torch.bfloat16)
    return W


def rms_hidden(T: int, H: int, device, seed: int):
    """Rows x / rms(x) with x ~ N(0,1), rounded to bf16."""
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(_stream_seed(seed, "hidden"))
    x = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
    x = x / torch.sqrt(torch.mean(x * x, dim=1, keepdim=True))
    return x.to(torch.bfloat16)


def topk_targets(hidden, W, seed: int, p_top: float = 0.9, k: int = 10):
    """Target ids: with prob ``p_top`` uniform among the row's top-``k`` scores, else uniform.

    The scores that rank candidate targets come from a plain bf16 torch matmul
    (cuBLAS, bf16 output) of the inputs; they only shape the target
    distribution and are never used as a logit anywhere.
    """
    torch = _torch()
    device = hidden.device
    T, V = hidden.shape[0], W.shape[0]
    g = torch.Generator(device=device)
    g.manual_seed(_stream_seed(seed, "targets"))
    top_idx = torch.empty((T, k), dtype=torch.int64, device=device)
    rows = 2048
    for r0 in range(0, T, rows):
        r1 = min(T, r0 + rows)
        scores = torch.matmul(hidden[r0:r1], W.t())
        top_idx[r0:r1] = torch.topk(scores, k, dim=1).indices
        del scores
    pick_top = torch.rand((T,), generator=g, device=device) < p_top
    which = torch.randint(0, k, (T,), generator=g, device=device)
    uniform = torch.randint(0, V, (T,), generator=g, device=device)
    chosen = torch.where(pick_top, top_idx.gather(1, which[:, None])[:, 0], uniform)
    return chosen.to(torch.int32)


@dataclass
class DeviceWorkload:
    """Device-resident inputs (torch tensors)."""
    name: str
    hidden: object              # torch.bfloat16 [T, H]
    W: object                   # torch.bfloat16 [V, H]
    targets: object             # torch.int32 [T]
    active: object = None       # torch.uint8 [T] or None
    n_shards: int = 1
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.hidden.shape[0])


def packed(W, device, T: int = 4096, seed: int = 1234) -> DeviceWorkload:
    """Packed training batch: 8 sequences x 512 tokens, all active, 4 shards."""
    hidden = rms_hidden(T, W.shape[1], device, seed)
    targets = topk_targets(hidden, W, seed)
    return DeviceWorkload("packed", hidden, W, targets, None, 4,
                          {"seed": seed, "seqs": T // 512, "seq_len": 512})


def decode_rows(T: int, n_source: int = 4096) -> np.ndarray:
    """Row indices of the packed batch used for a T-row decode batch (draw order)."""
    rng = _rng(1234 + T)
    return rng.choice(n_source, size=T, replace=False).astype(np.int64)


def grpo_long_layout(seed: int = 1235, prompts: int = 8, samples: int = 8,
                     prompt_len=(64, 512), resp_len=(256, 6912), chunk: int = 8192):
    """Sequence layout of the long-response GRPO batch.

    Returns (active mask uint8 [N], chunk boundaries list of (r0, r1), seq lengths).
    Each prompt's samples share its prompt length; prompt tokens are inactive,
    response tokens active; sequences are packed back to back and the stream
    is cut into ``chunk``-row calls (the last one ragged).
    """
    rng = _rng(seed)
    masks = []
    lens = []
    for _p in range(prompts):
        pl = int(rng.integers(prompt_len[0], prompt_len[1] + 1))
        for _s in range(samples):
            rl = int(rng.integers(resp_len[0], resp_len[1] + 1))
            masks.append(np.zeros(pl, dtype=np.uint8))
            masks.append(np.ones(rl, dtype=np.uint8))
            lens.append((pl, rl))
    active = np.concatenate(masks)
    n = active.shape[0]
    bounds = [(r0, min(n, r0 + chunk)) for r0 in range(0, n, chunk)]
    return active, bounds, lens


def grpo_long(W, device, seed: int = 1235) -> DeviceWorkload:
    torch = _torch()
    active, bounds, lens = grpo_long_layout(seed)
    hidden = rms_hidden(active.shape[0], W.shape[1], device, seed)
    targets = topk_targets(hidden, W, seed)
    return DeviceWorkload("grpo_long", hidden, W, targets,
                          torch.from_numpy(active).to(device), 4,
                          {"seed": seed, "chunks": bounds, "seq_lens": lens})


def sweep_set(W, device, T: int = 8192, seed: int = 1236) -> DeviceWorkload:
    hidden = rms_hidden(T, W.shape[1], device, seed)
    targets = topk_targets(hidden, W, seed)
    return DeviceWorkload("sweep", hidden, W, targets, None, 1, {"seed": seed})


def permutation(n: int, seed: int) -> np.ndarray:
    return _rng(seed).permutation(n).astype(np.int64)


# --------------------------------------------------------------------------
# numpy <-> torch helpers (pure data movement)
# --------------------------------------------------------------------------
def to_device(w: Workload, device) -> DeviceWorkload:
    torch = _torch()
    hid = torch.from_numpy(w.hidden.view(np.int16)).view(torch.bfloat16).to(device)
    W = torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16).to(device)
    tg = torch.from_numpy(w.targets).to(device)
    act = None if w.active is None else torch.from_numpy(w.active).to(device)
    return DeviceWorkload(w.name, hid, W, tg, act, w.n_shards, dict(w.meta))


def bf16_tensor_bits(t) -> np.ndarray:
    """A torch bf16 tensor (any device) as a numpy uint16 bit array."""
    torch = _torch()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def exact_device_case(T: int, H: int, V: int, device, seed: int, h_levels: int = 8,
                      w_levels: int = 4) -> DeviceWorkload:
    """Device-generated ``exact_case`` inputs at large sizes (hidden k/8, W j/64 grids)."""
    torch = _torch()
    assert H * h_levels * w_levels < (1 << 24)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    hid = (torch.randint(-h_levels, h_levels + 1, (T, H), generator=g, device=device)
           .to(torch.float32) / 8.0).to(torch.bfloat16)
    W = torch.empty((V, H), dtype=torch.bfloat16, device=device)
    rows = 8192
    for r0 in range(0, V, rows):
        r1 = min(V, r0 + rows)
        W[r0:r1] = (torch.randint(-w_levels, w_levels + 1, (r1 - r0, H), generator=g,
                                  device=device).to(torch.float32) / 64.0).to(torch.bfloat16)
    targets = torch.randint(0, V, (T,), generator=g, device=device).to(torch.int32)
    return DeviceWorkload("exact_device", hid, W, targets, None, 1, {"seed": seed, "exact": True})
