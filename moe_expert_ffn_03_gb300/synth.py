"""Seeded synthetic inputs for the grouped MXFP8 MoE expert FFN.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no routing, no quantization, no GEMM).  Both the CPU
oracle (through the tests) and the CUDA path receive the very same tensors
from it, so bit-exact comparisons never depend on two RNG implementations.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) evaluated at a counter, one independent
stream per (seed, tensor id).  Uniforms take the top 53 bits; normals come
from the Box-Muller transform in float64, are rounded to float32 and then to
bfloat16 (both round-to-nearest-even).  Everything is written with torch
integer/float ops so that the same code runs on the CPU and on a CUDA device.

Workload shapes follow the five expert-FFN workloads (tiny, uneven/Zipf,
Mixtral-8x7B-shaped forward, Mixtral-8x7B-shaped forward+backward, fine-grained
long-sequence); see ``configs.py``.
"""
from __future__ import annotations

import math

import torch

_GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1


def _s64(v: int) -> int:
    """Two's-complement view of an unsigned 64-bit constant (torch has no uint64 math)."""
    v &= _MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes (torch's >> is arithmetic)."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def splitmix64_py(state: int) -> int:
    """Reference scalar SplitMix64 output for a given (already advanced) state."""
    z = state & _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    """Base state of the stream for one tensor of one seed."""
    return splitmix64_py(((seed & 0xFFFFFFFF) << 32) | (tensor_id & 0xFFFFFFFF))


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(_M1)
    z = (z ^ _srl(z, 27)) * _s64(_M2)
    return z ^ _srl(z, 31)


def raw_u64(key: int, start: int, n: int, device) -> torch.Tensor:
    """SplitMix64 outputs for counters start..start+n-1 as int64 bit patterns."""
    ctr = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=device)
    z = ctr * _s64(_GAMMA) + _s64(key)
    return _mix(z)


def uniform(key: int, start: int, n: int, device) -> torch.Tensor:
    """float64 uniforms in the open interval (0, 1)."""
    top53 = _srl(raw_u64(key, start, n, device), 11)
    return (top53.to(torch.float64) + 0.5) * (2.0 ** -53)


_CHUNK = 1 << 24


def normal_f64(key: int, n: int, device, start: int = 0) -> torch.Tensor:
    """Standard normals (float64) for element indices start..start+n-1.

    Element 2i and 2i+1 of a stream are the Box-Muller pair built from the
    uniforms at counters 2i and 2i+1, so a value depends only on its index
    (chunking does not change the stream).  ``start`` must be even.
    """
    assert start % 2 == 0
    out = torch.empty(n, dtype=torch.float64, device=device)
    p_begin = start // 2
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, _CHUNK):
        p1 = min(npairs, p0 + _CHUNK)
        u = uniform(key, 2 * (p_begin + p0), 2 * (p1 - p0), device).view(-1, 2)
        r = torch.sqrt(-2.0 * torch.log(u[:, 0]))
        th = (2.0 * math.pi) * u[:, 1]
        z = torch.stack((r * torch.cos(th), r * torch.sin(th)), dim=1).reshape(-1)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo]
    return out


def normal_bf16(key: int, shape, std: float, device) -> torch.Tensor:
    """N(0, std^2) values: float64 normal * std, rounded to float32, then to bfloat16."""
    n = 1
    for s in shape:
        n *= s
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    step = _CHUNK * 4  # bounds the float64/int64 temporaries for full-size weights
    for s0 in range(0, n, step):
        s1 = min(n, s0 + step)
        z = normal_f64(key, s1 - s0, device, start=s0)
        out[s0:s1] = (z * std).to(torch.float32).to(torch.bfloat16)
    return out.view(*shape)


# tensor ids of the streams
TID_X, TID_LOGITS, TID_WGU, TID_WD, TID_DOUT, TID_BIAS, TID_WR = 1, 2, 3, 4, 5, 6, 7


def make_logits(cfg, seed: int, device) -> torch.Tensor:
    """Router logits [T][E] float32 with the workload's routing structure.

    * "normal":  N(0, 1) per entry (near-uniform expert loads).
    * "zipf":    Gumbel-top-k: logit = ln p_e + Gumbel(0, 1) with
                 p_e proportional to (e + 1)^-s for the first E-1 experts and
                 the last expert pinned to -1e30, so it receives no token.
    * "biased":  N(0, 1) + b_e with one bias b_e ~ N(0, bias_std^2) per expert.
    """
    T, E = cfg.T, cfg.E
    kind = cfg.routing
    if kind == "normal":
        z = normal_f64(stream_key(seed, TID_LOGITS), T * E, device).view(T, E)
        return z.to(torch.float32)
    if kind == "zipf":
        u = uniform(stream_key(seed, TID_LOGITS), 0, T * E, device).view(T, E)
        g = -torch.log(-torch.log(u))
        live = E - 1
        w = torch.tensor([(e + 1.0) ** (-cfg.zipf_s) for e in range(live)], dtype=torch.float64, device=device)
        lp = torch.log(w / w.sum())
        z = torch.empty(T, E, dtype=torch.float64, device=device)
        z[:, :live] = lp[None, :] + g[:, :live]
        z[:, live] = -1e30
        return z.to(torch.float32)
    if kind == "biased":
        z = normal_f64(stream_key(seed, TID_LOGITS), T * E, device).view(T, E)
        b = normal_f64(stream_key(seed, TID_BIAS), E, device) * cfg.bias_std
        return (z + b[None, :]).to(torch.float32)
    raise ValueError(f"unknown routing kind {kind!r}")


def make_inputs(cfg, seed: int = 0, device="cpu", with_grad: bool | None = None) -> dict:
    """All inputs of one workload: x, logits, W_gu, W_d and (for training) dout.

    Shapes: x [T][H] bf16 ~ N(0,1); logits [T][E] f32; W_gu [E][2I][H] bf16
    ~ N(0, 0.02^2) with rows 0..I-1 the gate and I..2I-1 the up projection;
    W_d [E][H][I] bf16 ~ N(0, 0.02^2); dout [T][H] bf16 ~ N(0, 0.01^2).
    """
    T, H, I, E = cfg.T, cfg.H, cfg.I, cfg.E
    if with_grad is None:
        with_grad = cfg.backward
    d = {
        "x": normal_bf16(stream_key(seed, TID_X), (T, H), 1.0, device),
        "logits": make_logits(cfg, seed, device),
        "w_gu": normal_bf16(stream_key(seed, TID_WGU), (E, 2 * I, H), cfg.w_std, device),
        "w_d": normal_bf16(stream_key(seed, TID_WD), (E, H, I), cfg.w_std, device),
    }
    if with_grad:
        d["dout"] = normal_bf16(stream_key(seed, TID_DOUT), (T, H), cfg.g_std, device)
    return d


def make_router_weight(cfg, seed: int = 0, device="cpu") -> torch.Tensor:
    """W_r [E][H] bf16 ~ N(0, 0.02^2) for the linear router."""
    return normal_bf16(stream_key(seed, TID_WR), (cfg.E, cfg.H), cfg.w_std, device)
