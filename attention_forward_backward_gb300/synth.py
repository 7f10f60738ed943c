"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only draws numbers. Both sides
receive the SAME arrays from here, so neither depends on the other.

Generator (a counter-based stream, written from its published definitions):

* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): output n of the stream with state ``seed`` is
  ``mix(seed + (n + 1) * 0x9E3779B97F4A7C15)`` with the Stafford "Mix13"
  finaliser (shifts 30/27/31, multipliers 0xBF58476D1CE4E5B9 and
  0x94D049BB133111EB).
* A uniform double in [0, 1) is the top 53 bits of an output times 2^-53.
* Element n of a tensor is one Box-Muller normal (Box & Muller 1958) from the
  outputs 2n and 2n+1: ``sqrt(-2 ln(1 - u0)) * cos(2 pi u1)``, computed in
  float64 and rounded once to float32 (round to nearest even).
* Flat element order is the row-major order of [B, H, L, D].
* Seeds: ``1000 * cfg + tensor_id`` with Q = 0, K = 1, V = 2, dO = 3.

bf16 inputs (the accelerated contract) are the float32 values rounded to
bfloat16 with IEEE round-to-nearest-even on the bit pattern, done here so that
the GPU and the oracle get bit-identical operands.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_IDS = {"Q": 0, "K": 1, "V": 2, "dO": 3}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the SplitMix64 stream for ``seed``."""
    n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + n * _GAMMA
        return _mix(z)


def normal_f32(seed: int, count: int, chunk: int = 1 << 22) -> np.ndarray:
    """``count`` standard normals as float32, element n from outputs 2n, 2n+1."""
    out = np.empty(count, dtype=np.float32)
    two_pi = 2.0 * math.pi
    for s in range(0, count, chunk):
        c = min(chunk, count - s)
        r = splitmix64(seed, 2 * s, 2 * c).reshape(c, 2)
        u = (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        rad = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
        out[s:s + c] = (rad * np.cos(two_pi * u[:, 1])).astype(np.float32)
    return out


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bfloat16 (ties to even); returns the uint16
    bit patterns. Inputs here are finite normals, so no NaN handling is needed."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_f16(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest IEEE half (ties to even, numpy's conversion);
    returns the uint16 bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def base_contract(contract: str) -> str:
    """"strict", "accel" or "accel_f16": the input format of a contract name
    ("+out16" and other suffixes name output options, not input formats)."""
    return contract.split("+")[0]


def encode(x: np.ndarray, contract: str):
    """Host input in the contract's format: f32 array (strict), or the 16-bit bit
    patterns (key "bits") with their exact float32 values (key "values") that the
    oracle consumes: bf16 (accel) or f16 (accel_f16), rounded to nearest even."""
    c = base_contract(contract)
    if c == "strict":
        return x
    if c == "accel":
        bits = round_to_bf16(x)
        return {"bits": bits, "values": bf16_bits_to_f32(bits)}
    if c == "accel_f16":
        bits = round_to_f16(x)
        return {"bits": bits, "values": f16_bits_to_f32(bits)}
    raise ValueError(contract)


@dataclass(frozen=True)
class Workload:
    """One seeded attention workload. Shapes are [B, H, L, D] row-major."""
    cfg: int
    B: int
    H: int
    L: int
    D: int
    causal: bool
    contracts: tuple
    qk_gain: float = 1.0
    name: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def shape(self):
        return (self.B, self.H, self.L, self.D)

    @property
    def numel(self) -> int:
        return self.B * self.H * self.L * self.D

    def flops_fwd(self) -> float:
        """4 B H L^2 D, halved when causal (the convention the throughput
        numbers are quoted in; not L(L+1)/2)."""
        f = 4.0 * self.B * self.H * self.L * self.L * self.D
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


# The five workloads. Scale is 1/sqrt(D) everywhere; cfg 4 multiplies the Q
# and K draws by 4 so that logits have standard deviation 16.
WORKLOADS = {
    1: Workload(1, 1, 2, 64, 32, True, ("strict",), name="tiny causal B1 H2 L64 D32"),
    2: Workload(2, 4, 8, 512, 64, True, ("strict", "accel"), name="decoder causal B4 H8 L512 D64"),
    3: Workload(3, 32, 12, 197, 64, False, ("accel",), name="encoder full B32 H12 L197 D64"),
    4: Workload(4, 8, 16, 2048, 64, True, ("strict", "accel"), qk_gain=4.0,
                name="large-logit causal B8 H16 L2048 D64 (Q,K x4)"),
    5: Workload(5, 2, 32, 8192, 128, True, ("strict", "accel"),
                name="long-sequence causal B2 H32 L8192 D128"),
}


def tensor_f32(w: Workload, which: str) -> np.ndarray:
    """Seeded float32 tensor ``which`` in {Q, K, V, dO} of workload ``w``."""
    seed = 1000 * w.cfg + TENSOR_IDS[which]
    x = normal_f32(seed, w.numel).reshape(w.shape)
    if which in ("Q", "K") and w.qk_gain != 1.0:
        x *= np.float32(w.qk_gain)
    return x


def inputs(w: Workload, contract: str):
    """Dict of host inputs for a contract.

    strict -> float32 arrays. accel (accel_f16) -> uint16 bf16 (f16) bit
    patterns (key "bits") plus their exact float32 values (key "values"), which
    the oracle consumes.
    """
    return {t: encode(tensor_f32(w, t), contract) for t in ("Q", "K", "V", "dO")}


def custom_workload(B, H, L, D, causal, seed_cfg=900, qk_gain=1.0) -> Workload:
    """An ad-hoc workload (edge cases in tests) with its own seed block."""
    return Workload(seed_cfg, B, H, L, D, bool(causal), ("strict", "accel"), qk_gain,
                    name=f"custom B{B} H{H} L{L} D{D} {'causal' if causal else 'full'}")


def cross_inputs(B, H, Lq, Lk, D, contract: str, seed_cfg: int = 950):
    """Seeded inputs with Lq query rows and Lk key rows (cross attention): Q and
    dO are [B, H, Lq, D], K and V [B, H, Lk, D]; same generator, seeds and
    formats as ``inputs``."""
    out = {}
    for t in ("Q", "K", "V", "dO"):
        rows = Lq if t in ("Q", "dO") else Lk
        x = normal_f32(1000 * seed_cfg + TENSOR_IDS[t], B * H * rows * D).reshape(B, H, rows, D)
        out[t] = encode(x, contract)
    return out


# ---------------------------------------------------------------- convolution layers
CONV_TENSOR_IDS = {"X": 4, "Wt": 5, "dY": 6}


@dataclass(frozen=True)
class ConvWorkload:
    """One seeded 2-D convolution layer, channels last: X [N, H, W, C], Wt
    [K, R, S, C], dY [N, P, Q, K] with P = (H + 2 pad - R) // stride + 1."""
    cid: int
    N: int
    H: int
    W: int
    C: int
    K: int
    R: int
    S: int
    stride: int
    pad: int
    name: str = ""

    @property
    def P(self) -> int:
        return (self.H + 2 * self.pad - self.R) // self.stride + 1

    @property
    def Q(self) -> int:
        return (self.W + 2 * self.pad - self.S) // self.stride + 1

    def shapes(self):
        return {"X": (self.N, self.H, self.W, self.C), "Wt": (self.K, self.R, self.S, self.C),
                "dY": (self.N, self.P, self.Q, self.K)}

    def flops(self) -> float:
        """2 N P Q K C R S: one derivative (input or weight gradient)."""
        return 2.0 * self.N * self.P * self.Q * self.K * self.C * self.R * self.S

    def with_batch(self, N: int) -> "ConvWorkload":
        return ConvWorkload(self.cid, N, self.H, self.W, self.C, self.K, self.R, self.S,
                            self.stride, self.pad, self.name.replace(f"N{self.N}", f"N{N}"))


def _resnet(cid, H, C, K, R, stride, pad, what, N=32):
    P = (H + 2 * pad - R) // stride + 1
    return ConvWorkload(cid, N, H, H, C, K, R, R, stride, pad,
                        name=f"{what} {R}x{R}/{stride} {C}->{K} {H}->{P} N{N}")


# The distinct convolution shapes of a ResNet-50 (v1.5: stride on the 3x3 of the
# first block of a stage) on 224 x 224 images, batch 32; the stem (C = 3) is
# left out (see the derivative functions' channel rule).
CONV_WORKLOADS = {
    1: _resnet(1, 56, 64, 64, 3, 1, 1, "res2 3x3"),
    2: _resnet(2, 56, 256, 64, 1, 1, 0, "res2 reduce"),
    3: _resnet(3, 56, 64, 256, 1, 1, 0, "res2 expand"),
    4: _resnet(4, 56, 128, 128, 3, 2, 1, "res3 3x3 strided"),
    5: _resnet(5, 28, 128, 128, 3, 1, 1, "res3 3x3"),
    6: _resnet(6, 56, 256, 512, 1, 2, 0, "res3 downsample"),
    7: _resnet(7, 14, 256, 256, 3, 1, 1, "res4 3x3"),
    8: _resnet(8, 14, 1024, 256, 1, 1, 0, "res4 reduce"),
    9: _resnet(9, 7, 512, 512, 3, 1, 1, "res5 3x3"),
    10: _resnet(10, 7, 512, 2048, 1, 1, 0, "res5 expand"),
}


def conv_tensor_f32(w: ConvWorkload, which: str) -> np.ndarray:
    """Seeded float32 tensor ``which`` in {X, Wt, dY}: X = |normal| (activations
    after a ReLU), Wt = normal * sqrt(2 / (C R S)) (He initialisation), dY =
    normal."""
    shape = w.shapes()[which]
    seed = 1000 * (100 + w.cid) + CONV_TENSOR_IDS[which]
    x = normal_f32(seed, int(np.prod(shape))).reshape(shape)
    if which == "X":
        x = np.abs(x)
    elif which == "Wt":
        x *= np.float32(math.sqrt(2.0 / (w.C * w.R * w.S)))
    return x


def conv_inputs(w: ConvWorkload, contract: str = "accel"):
    """Host inputs X, Wt, dY of a convolution layer in a 16-bit contract's format
    (bit patterns and their exact float32 values, as ``encode``)."""
    return {t: encode(conv_tensor_f32(w, t), contract) for t in ("X", "Wt", "dY")}


def custom_conv(N, H, W, C, K, R, S, stride, pad, cid=200) -> ConvWorkload:
    """An ad-hoc convolution (edge cases in tests) with its own seed block."""
    return ConvWorkload(cid, N, H, W, C, K, R, S, stride, pad,
                        name=f"custom N{N} {H}x{W} {C}->{K} {R}x{S}/{stride} pad{pad}")
