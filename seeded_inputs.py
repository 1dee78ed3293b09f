"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module only draws numbers. It holds none of the attention arithmetic, so
both the CPU oracle and the CUDA path can take their inputs from here without
sharing any of the computation under test.

Generator (counter-based, so any element can be drawn independently):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) in its counter form: word ``n`` of a stream with
  state ``s0`` is ``mix64(s0 + (n + 1) * GAMMA)`` with
  ``GAMMA = 0x9E3779B97F4A7C15`` and ``mix64`` the SplitMix64 finaliser.
* A stream is keyed by ``(seed, tensor_id)``:
  ``s0 = mix64(seed * GAMMA + tensor_id)``.
* Uniforms on the open interval (0, 1): ``((w >> 11) + 0.5) * 2**-53``.
* Standard normals by Box-Muller (1958) in float64: element pair ``m`` uses
  words ``2m`` and ``2m + 1``; ``r = sqrt(-2 ln u1)``, ``theta = 2 pi u2``;
  element ``2m`` is ``r cos theta`` and element ``2m + 1`` is ``r sin theta``.
* bf16 values: the float64 normal is rounded to float32 (round to nearest
  even), then to bf16 (round to nearest even).  A multiplier that is a power
  of two (the peaked and long-context workloads) is applied to the bf16 value
  exactly, so every consumer sees the same bits.

Tensors are returned as ``numpy.uint16`` arrays of bf16 bit patterns, laid out
``[B][H][S][D]`` row-major.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Tensor ids of the streams drawn for one workload.
TID_Q, TID_K, TID_V, TID_ROWS = 1, 2, 3, 4

_CHUNK = 1 << 22  # elements drawn per vectorised chunk (bounds temporaries)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_state(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) * GAMMA + np.uint64(tensor_id)
        return _mix64(s)[0]


def uniform_words(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of stream (seed, tensor_id) as uint64."""
    s0 = _stream_state(seed, tensor_id)
    n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(s0 + n * GAMMA)


def _words_to_unit(w: np.ndarray) -> np.ndarray:
    return ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal_f64(seed: int, tensor_id: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` standard normals (float64) from element ``start`` of the stream.

    ``start`` must be even so that Box-Muller pairs line up.
    """
    if start % 2:
        raise ValueError("start must be even")
    npairs = (count + 1) // 2
    w = uniform_words(seed, tensor_id, start, 2 * npairs)
    u1 = _words_to_unit(w[0::2])
    u2 = _words_to_unit(w[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    th = (2.0 * math.pi) * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)
    return out[:count]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even); returns uint16 bit patterns.

    Inputs here are finite; NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 exactly."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, tensor_id: int, count: int, multiplier: float = 1.0) -> np.ndarray:
    """``count`` N(0,1) draws rounded to bf16, times an exact power of two."""
    if multiplier != 1.0:
        m, e = math.frexp(multiplier)
        if m != 0.5:
            raise ValueError("multiplier must be a power of two")
    out = np.empty(count, dtype=np.uint16)
    for lo in range(0, count, _CHUNK):
        n = min(_CHUNK, count - lo)
        x = normal_f64(seed, tensor_id, n, start=lo).astype(np.float32)
        bits = f32_to_bf16_bits(x)
        if multiplier != 1.0:
            bits = f32_to_bf16_bits(bf16_bits_to_f32(bits) * np.float32(multiplier))
        out[lo:lo + n] = bits
    return out


def qkv_bf16(seed: int, B: int, H: int, S_q: int, S_kv: int, D: int,
             q_mult: float = 1.0, k_mult: float = 1.0):
    """Q, K, V of one workload as uint16 bf16 bits, shapes [B,H,S,D]."""
    q = normal_bf16(seed, TID_Q, B * H * S_q * D, q_mult).reshape(B, H, S_q, D)
    k = normal_bf16(seed, TID_K, B * H * S_kv * D, k_mult).reshape(B, H, S_kv, D)
    v = normal_bf16(seed, TID_V, B * H * S_kv * D).reshape(B, H, S_kv, D)
    return q, k, v


def sample_rows(seed: int, S: int, n: int, must_include=()) -> np.ndarray:
    """``n`` distinct row indices in [0, S) (sorted), always holding ``must_include``.

    Rows come from stream (seed, TID_ROWS): a partial Fisher-Yates shuffle of
    0..S-1 driven by its words.
    """
    n = min(n, S)
    chosen = [r for r in dict.fromkeys(int(r) for r in must_include) if 0 <= r < S]
    pool = {}
    words = uniform_words(seed, TID_ROWS, 0, S if S < 4 * n else 4 * n)
    picked = set(chosen)
    wi = 0
    i = 0
    while len(chosen) < n:
        # swap position i with a uniform j in [i, S)
        j = i + int(words[wi % len(words)] % np.uint64(S - i))
        wi += 1
        vi, vj = pool.get(i, i), pool.get(j, j)
        pool[i], pool[j] = vj, vi
        i += 1
        if vj not in picked:
            picked.add(vj)
            chosen.append(vj)
        if i >= S:
            break
    return np.array(sorted(chosen[:n]), dtype=np.int64)


# --- the same generator on a torch device (bench inputs at full size) --------

def _to_i64(x: int) -> int:
    x &= (1 << 64) - 1
    return x - (1 << 64) if x >= (1 << 63) else x


def _lsr_t(z, k: int):
    """Logical right shift of an int64 tensor viewed as uint64."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix64_t(z):
    z = (z ^ _lsr_t(z, 30)) * _to_i64(0xBF58476D1CE4E5B9)
    z = (z ^ _lsr_t(z, 27)) * _to_i64(0x94D049BB133111EB)
    return z ^ _lsr_t(z, 31)


def _mix64_int(z: int) -> int:
    m = (1 << 64) - 1
    z &= m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def normal_bf16_torch(seed: int, tensor_id: int, count: int, multiplier: float = 1.0,
                      device="cuda", chunk: int = 1 << 25):
    """Same definition as ``normal_bf16`` computed with torch on ``device``.

    Returns a bfloat16 tensor of ``count`` elements.  The float64 log, sqrt,
    cos and sin of the device may differ from the host's in the last place,
    which can move a value by one bf16 step in rare cases; parity tests
    therefore draw on the host, and this path serves the benchmark.
    """
    import torch

    if multiplier != 1.0 and math.frexp(multiplier)[0] != 0.5:
        raise ValueError("multiplier must be a power of two")
    s0 = _mix64_int(seed * 0x9E3779B97F4A7C15 + tensor_id)
    gamma = _to_i64(0x9E3779B97F4A7C15)
    out = torch.empty(count, dtype=torch.bfloat16, device=device)
    for lo in range(0, count, chunk):
        n = min(chunk, count - lo)
        npairs = (n + 1) // 2
        idx = torch.arange(lo + 1, lo + 2 * npairs + 1, dtype=torch.int64, device=device)
        w = _mix64_t(idx * gamma + _to_i64(s0))
        u = (_lsr_t(w, 11).to(torch.float64) + 0.5) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = torch.sqrt(-2.0 * torch.log(u1))
        th = (2.0 * math.pi) * u2
        z = torch.stack([r * torch.cos(th), r * torch.sin(th)], dim=1).reshape(-1)[:n]
        x = z.to(torch.float32).to(torch.bfloat16)
        if multiplier != 1.0:
            x = x * multiplier
        out[lo:lo + n] = x
    return out


def qkv_bf16_torch(seed: int, B: int, H: int, S_q: int, S_kv: int, D: int,
                   q_mult: float = 1.0, k_mult: float = 1.0, device="cuda"):
    """Q, K, V of one workload as bf16 tensors [B,H,S,D] on ``device``."""
    q = normal_bf16_torch(seed, TID_Q, B * H * S_q * D, q_mult, device).view(B, H, S_q, D)
    k = normal_bf16_torch(seed, TID_K, B * H * S_kv * D, k_mult, device).view(B, H, S_kv, D)
    v = normal_bf16_torch(seed, TID_V, B * H * S_kv * D, 1.0, device).view(B, H, S_kv, D)
    return q, k, v


# --- e4m3 (FP8) inputs ---------------------------------------------------------
#
# e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 holds
# the subnormals m * 2^-9; the largest finite magnitude is 448 and code 0x7F
# (with either sign) is NaN.  Every e4m3 value is exactly a bf16 value, so the
# bf16 oracle sees the e4m3 inputs without rounding.

def _e4m3_magnitudes() -> np.ndarray:
    vals = np.empty(128, dtype=np.float64)
    for code in range(128):
        e, m = code >> 3, code & 7
        vals[code] = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    vals[127] = np.nan
    return vals


E4M3_MAGNITUDES = _e4m3_magnitudes()  # codes 0..126 finite and increasing
E4M3_MAX = 448.0


def f64_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even code), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    t = E4M3_MAGNITUDES[:127]
    hi = np.clip(np.searchsorted(t, a), 1, 126)
    lo = hi - 1
    d_lo = a - t[lo]
    d_hi = t[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) << np.uint8(7))


def e4m3_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen e4m3 codes to float32 exactly."""
    bits = np.asarray(bits, dtype=np.uint8)
    mag = E4M3_MAGNITUDES[bits & np.uint8(0x7F)]
    return np.where(bits & np.uint8(0x80), -mag, mag).astype(np.float32)


def e4m3_bits_to_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """The same values as bf16 bit patterns (exact: e4m3 is a subset of bf16)."""
    return f32_to_bf16_bits(e4m3_bits_to_f32(bits))


def normal_e4m3(seed: int, tensor_id: int, count: int, multiplier: float = 1.0) -> np.ndarray:
    """``count`` draws of N(0,1) * multiplier rounded to e4m3 (uint8 codes)."""
    out = np.empty(count, dtype=np.uint8)
    for lo in range(0, count, _CHUNK):
        n = min(_CHUNK, count - lo)
        out[lo:lo + n] = f64_to_e4m3_bits(normal_f64(seed, tensor_id, n, start=lo) * multiplier)
    return out


def qkv_e4m3(seed: int, B: int, H: int, S_q: int, S_kv: int, D: int,
             mults=(1.0, 1.0, 1.0)):
    """Q, K, V as e4m3 codes [B,H,S,D]; element = round(N(0,1) * mult)."""
    q = normal_e4m3(seed, TID_Q, B * H * S_q * D, mults[0]).reshape(B, H, S_q, D)
    k = normal_e4m3(seed, TID_K, B * H * S_kv * D, mults[1]).reshape(B, H, S_kv, D)
    v = normal_e4m3(seed, TID_V, B * H * S_kv * D, mults[2]).reshape(B, H, S_kv, D)
    return q, k, v


def normal_e4m3_torch(seed: int, tensor_id: int, count: int, multiplier: float = 1.0, device="cuda",
                      chunk: int = 1 << 25):
    """Device version for the benchmark: the same normals, rounded through
    float32 to torch.float8_e4m3fn (a float32 tie can round differently from
    the host's direct rounding in rare cases; parity tests draw on the host)."""
    import torch

    out = torch.empty(count, dtype=torch.float8_e4m3fn, device=device)
    for lo in range(0, count, chunk):
        n = min(chunk, count - lo)
        # the bf16 draw holds the same float64 normal rounded twice; redo it in float32
        npairs = (n + 1) // 2
        s0 = _mix64_int(seed * 0x9E3779B97F4A7C15 + tensor_id)
        idx = torch.arange(lo + 1, lo + 2 * npairs + 1, dtype=torch.int64, device=device)
        w = _mix64_t(idx * _to_i64(0x9E3779B97F4A7C15) + _to_i64(s0))
        u = (_lsr_t(w, 11).to(torch.float64) + 0.5) * (2.0 ** -53)
        r = torch.sqrt(-2.0 * torch.log(u[0::2]))
        th = (2.0 * math.pi) * u[1::2]
        z = torch.stack([r * torch.cos(th), r * torch.sin(th)], dim=1).reshape(-1)[:n] * multiplier
        out[lo:lo + n] = z.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float32).to(torch.float8_e4m3fn)
    return out
