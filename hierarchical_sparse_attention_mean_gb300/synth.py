"""Seeded synthetic inputs for LLSA: the one module both the CUDA path's tests
and the CPU oracle's tests draw from. It holds none of the method's arithmetic.

Random numbers: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style: the value
for counter c of stream `key` is mix(key + (c + 1) * 0x9E3779B97F4A7C15), where
mix is SplitMix64's finaliser. Normal deviates come from Box-Muller on pairs of
counters (2m, 2m+1), each mapped to a uniform in (0, 1) as ((z >> 11) + 0.5) /
2^53. Stream keys are derived from (seed, tensor id, slice index) so that every
(batch, head) slice can be generated independently and in parallel.

Workloads (raster token order, B = 16):
  * iid inputs: Q, K, V ~ N(0, 1) * amplitude, dO ~ N(0, 1).
  * pixel-DiT stand-ins: per slice, one latent 2D Gaussian random field F with
    d channels on the H x W pixel grid (white N(0, 1) noise convolved with a
    separable Gaussian of standard deviation `length_scale` pixels, truncated at
    4 sigma, periodic boundary, then scaled to unit RMS per channel), and
    Q = F + 0.3 N(0, 1), K = F + 0.3 N(0, 1) with independent noise; V and dO
    iid N(0, 1). Q and K sharing one field gives block scores the spatial
    locality that attention maps of images show.
Values are rounded to bf16 (round to nearest even) for bf16 workloads, so the
float32 arrays returned hold exactly what the GPU receives.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids of the streams
Q_ID, K_ID, V_ID, DO_ID, FIELD_ID, QNOISE_ID, KNOISE_ID = range(7)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_int(x: int) -> int:
    with np.errstate(over="ignore"):
        return int(_mix(np.array([x % (1 << 64)], np.uint64))[0])


def stream_key(seed: int, tensor_id: int, slice_index: int) -> int:
    """Key of the counter stream for one tensor of one (batch, head) slice."""
    return _mix_int(_mix_int(seed) ^ ((tensor_id << 40) + slice_index))


def uint64_stream(key: int, start: int, count: int) -> np.ndarray:
    """SplitMix64 outputs for counters start .. start+count-1 of stream key."""
    c = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + c * _GOLDEN)


def normal(key: int, count: int) -> np.ndarray:
    """count standard normal deviates (float64) of stream key via Box-Muller."""
    pairs = (count + 1) // 2
    z = uint64_stream(key, 0, 2 * pairs)
    u = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * pairs, np.float64)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out[:count]


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); returns float32."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def gaussian_field(key: int, H: int, W: int, d: int, length_scale: float) -> np.ndarray:
    """Latent field [H*W, d] (raster rows), unit RMS per channel."""
    white = normal(key, d * H * W).reshape(d, H, W)
    R = int(math.floor(4.0 * length_scale))
    off = np.arange(-R, R + 1)
    g = np.exp(-0.5 * (off / length_scale) ** 2)
    gx = np.zeros(W)
    np.add.at(gx, off % W, g)
    gy = np.zeros(H)
    np.add.at(gy, off % H, g)
    kern = np.fft.rfft2(np.outer(gy, gx))
    f = np.fft.irfft2(np.fft.rfft2(white) * kern, s=(H, W))
    f /= np.sqrt(np.mean(f * f, axis=(1, 2), keepdims=True))
    return np.ascontiguousarray(f.reshape(d, H * W).T)


@dataclass(frozen=True)
class Workload:
    """One synthetic LLSA workload. `name` says what it is with its sizes."""
    name: str
    batch: int
    heads: int
    n: int
    d: int
    block: int = 16
    topk: int = 8
    dtype: str = "bf16"           # "bf16" or "fp32"
    kind: str = "iid"             # "iid" or "grf"
    amplitude: float = 1.0        # scale of iid Q, K, V
    length_scale: float = 8.0     # GRF standard deviation, pixels
    grid: tuple = field(default=(0, 0))  # (H, W) pixel grid, raster order
    seed: int = 1000
    backward: bool = True

    @property
    def bh(self) -> int:
        return self.batch * self.heads


WORKLOADS = {
    w.name: w for w in [
        Workload("llsa-fwd-n1024-d64-b1h1-K4-fp32", 1, 1, 1024, 64, topk=4, dtype="fp32",
                 grid=(32, 32), seed=1001, backward=False),
        Workload("llsa-fwd-n4096-d64-b2h8-K8-bf16", 2, 8, 4096, 64, amplitude=0.5, grid=(64, 64),
                 seed=1002, backward=False),
        Workload("llsa-n16384-d64-b2h12-K8-bf16", 2, 12, 16384, 64, amplitude=0.5, grid=(128, 128),
                 seed=1003),
        Workload("llsa-n65536-d64-b1h12-K8-grf8-bf16", 1, 12, 65536, 64, kind="grf", length_scale=8.0,
                 grid=(256, 256), seed=1004),
        Workload("llsa-n262144-d128-b1h16-K16-grf16-bf16", 1, 16, 262144, 128, topk=16, kind="grf",
                 length_scale=16.0, grid=(512, 512), seed=1005),
    ]
}
# the workload the throughput figure is quoted on: 256x256 pixel tokens
HEADLINE = "llsa-n65536-d64-b1h12-K8-grf8-bf16"


def make_slice(w: Workload, s: int, with_dout: bool = True) -> dict:
    """Inputs of (batch, head) slice s: float32 arrays [n, d] (bf16-exact for
    bf16 workloads)."""
    n, d = w.n, w.d
    rnd = bf16_round if w.dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    out = {}
    if w.kind == "grf":
        H, W = w.grid
        assert H * W == n, "grid must cover the tokens"
        f = gaussian_field(stream_key(w.seed, FIELD_ID, s), H, W, d, w.length_scale)
        out["q"] = rnd(f + 0.3 * normal(stream_key(w.seed, QNOISE_ID, s), n * d).reshape(n, d))
        out["k"] = rnd(f + 0.3 * normal(stream_key(w.seed, KNOISE_ID, s), n * d).reshape(n, d))
        out["v"] = rnd(normal(stream_key(w.seed, V_ID, s), n * d).reshape(n, d))
    else:
        a = w.amplitude
        out["q"] = rnd(a * normal(stream_key(w.seed, Q_ID, s), n * d).reshape(n, d))
        out["k"] = rnd(a * normal(stream_key(w.seed, K_ID, s), n * d).reshape(n, d))
        out["v"] = rnd(a * normal(stream_key(w.seed, V_ID, s), n * d).reshape(n, d))
    if with_dout:
        out["dout"] = rnd(normal(stream_key(w.seed, DO_ID, s), n * d).reshape(n, d))
    return out


def make_inputs(w: Workload, with_dout: bool = True, slices=None, threads: int = 8) -> dict:
    """Inputs of the listed slices (all by default): float32 [len, n, d] each."""
    idx = list(range(w.bh)) if slices is None else list(slices)
    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        parts = list(ex.map(lambda s: make_slice(w, s, with_dout), idx))
    return {key: np.stack([p[key] for p in parts]) for key in parts[0]}


def small(name: str, batch: int, heads: int, n: int, d: int, block: int = 16, topk: int = 8,
          dtype: str = "bf16", amplitude: float = 0.5, seed: int = 7) -> Workload:
    """An ad-hoc iid workload for tests (ragged tails, edge cases)."""
    side = int(math.isqrt(n))
    grid = (side, side) if side * side == n else (1, n)
    return Workload(name, batch, heads, n, d, block=block, topk=topk, dtype=dtype, amplitude=amplitude,
                    grid=grid, seed=seed)
