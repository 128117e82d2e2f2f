"""Seeded synthetic workloads for the quantized paged KV store.

This module is shared by both sides of every parity check (the CPU oracle and
the CUDA library) and by the benchmark.  It contains random draws, workload
shapes and page-table construction only: no quantization, dequantization or
attention arithmetic.  The one derived quantity it computes is the workload's
calibration recipe for the scale inputs (per-tensor amax divided by the
format's largest value), which both sides then receive as plain inputs.

Value distributions follow "KV cache quantization: mechanism and traps"
(hrletsgo.me), section "Why K and V distributions differ": keys carry
per-channel outliers (a few head_dim channels with much larger magnitude),
values vary per token.  Shapes follow the Llama-3-8B layer (32 q heads, 8 kv
heads, head_dim 128) and the Llama-3-70B layer (64 q heads, 8 kv heads,
head_dim 128) of the same page's "INT8, FP8, INT4: measured numbers" section,
with page size 16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

# Largest finite magnitude of each format, used only by the calibration
# recipe (amax / max).  E4M3 is the "fn" variant (448); E5M2 57344; NVFP4's
# global scale divides by 448 * 6 = 2688 (FP8 block-scale max times E2M1 max).
_CAL_DIVISOR = {"fp8_e4m3": 448.0, "fp8_e5m2": 57344.0, "nvfp4": 2688.0}

FORMAT_NAMES = ("bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4")


def _gen(seed: int, *stream: int) -> torch.Generator:
    """Independent CPU generator for (seed, stream ids)."""
    h = seed & 0xFFFFFFFF
    for s in stream:
        h = (h * 1_000_003 + s * 7919 + 12345) % (2**61 - 1)
    return torch.Generator().manual_seed(h)


def to_bf16_bits(x: torch.Tensor) -> np.ndarray:
    """float32 tensor -> numpy uint16 bfloat16 bit patterns (round to nearest even)."""
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_float(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    """One layer stack of a decode workload.

    Token t of sequence b is stored at slot page_table[b][t // P] * P + t % P.
    K/V for a (layer, sequence) are regenerated on demand from the seed, so a
    full-size workload never has to be held in host memory at once.
    """
    name: str
    fmt: str
    layers: int
    Hq: int
    Hkv: int
    D: int
    P: int
    seq_lens: np.ndarray          # int32 [B]
    page_table: np.ndarray        # int32 [B][max_pages], -1 past the end
    num_pages: int
    seed: int
    k_outlier_channels: int
    k_outlier_lo: float
    k_outlier_hi: float
    v_std: float
    v_token_sigma: float          # 0: no per-token scale
    scale_mode: str = "amax"      # "amax" or "one" (the default-1.0 case)
    sm_scale: float = 0.0
    _scales: dict = dataclasses.field(default_factory=dict)

    def __post_init__(self):
        if not self.sm_scale:
            self.sm_scale = 1.0 / math.sqrt(self.D)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.seq_lens.sum())

    # ---- draws ------------------------------------------------------------
    def q(self, layer: int = 0, step: int = 0) -> np.ndarray:
        """bf16 bits [B][Hq][D], N(0, 1)."""
        g = _gen(self.seed, 1, layer, step)
        return to_bf16_bits(torch.randn(self.B, self.Hq, self.D, generator=g))

    def _outliers(self, layer: int):
        g = _gen(self.seed, 2, layer)
        chans = torch.stack([torch.randperm(self.D, generator=g)[: self.k_outlier_channels]
                             for _ in range(self.Hkv)])
        fac = self.k_outlier_lo + (self.k_outlier_hi - self.k_outlier_lo) * torch.rand(
            self.Hkv, self.k_outlier_channels, generator=g)
        mult = torch.ones(self.Hkv, self.D)
        for h in range(self.Hkv):
            mult[h, chans[h]] = fac[h]
        return mult

    def kv_float(self, layer: int, b: int, t0: int = 0, t1: int | None = None):
        """float32 K, V [t1 - t0][Hkv][D] for tokens [t0, t1) of sequence b (before bf16)."""
        T = int(self.seq_lens[b])
        t1 = T if t1 is None else t1
        g = _gen(self.seed, 3, layer, b)
        # draw the whole sequence so that any token range gives identical values
        k = torch.randn(T, self.Hkv, self.D, generator=g)
        v = torch.randn(T, self.Hkv, self.D, generator=g) * self.v_std
        if self.v_token_sigma > 0:
            z = torch.randn(T, self.Hkv, 1, generator=g)
            v = v * torch.exp(self.v_token_sigma * z)
        k = k * self._outliers(layer)
        return k[t0:t1], v[t0:t1]

    def kv(self, layer: int, b: int, t0: int = 0, t1: int | None = None):
        """bf16 bits K, V [t1 - t0][Hkv][D]."""
        k, v = self.kv_float(layer, b, t0, t1)
        return to_bf16_bits(k), to_bf16_bits(v)

    def slots(self, b: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
        T = int(self.seq_lens[b])
        t1 = T if t1 is None else t1
        t = np.arange(t0, t1, dtype=np.int64)
        return self.page_table[b, t // self.P].astype(np.int64) * self.P + t % self.P

    # ---- calibration recipe (an input to both sides) -----------------------
    def kv_all(self, layer: int = 0):
        """bf16 bits K, V of every sequence (two lists), drawn once; also fixes
        the layer's scale inputs from them."""
        ks, vs = [], []
        for b in range(self.B):
            k, v = self.kv(layer, b)
            ks.append(k)
            vs.append(v)
        if layer not in self._scales:
            amax = self._scales.setdefault(("amax", layer), self._amax_of(ks, vs))
            self._scales[layer] = self._scales_of(amax)
        return ks, vs

    def _scales_from(self, ks, vs, fmt=None) -> np.ndarray:
        return self._scales_of(self._amax_of(ks, vs), fmt)

    @staticmethod
    def _amax_of(ks, vs):
        ka = max((float(np.abs(bf16_bits_to_float(k)).max()) for k in ks if k.size), default=0.0)
        va = max((float(np.abs(bf16_bits_to_float(v)).max()) for v in vs if v.size), default=0.0)
        return ka, va

    def _scales_of(self, amax, fmt=None) -> np.ndarray:
        div = _CAL_DIVISOR.get(fmt or self.fmt)
        if div is None or self.scale_mode == "one":
            return np.ones(2, np.float32)
        ka, va = amax
        return np.array([ka / div if ka > 0 else 1.0, va / div if va > 0 else 1.0], np.float32)

    def scales_for(self, fmt: str, ks, vs, layer: int = 0) -> np.ndarray:
        """The scale inputs the calibration recipe gives format `fmt` on this
        layer's rows ks, vs (the per-tensor amax is computed once per layer)."""
        key = ("amax", layer)
        if key not in self._scales:
            self._scales[key] = self._amax_of(ks, vs)
        return self._scales_of(self._scales[key], fmt)

    def q_scales(self, layer: int = 0, per_head: bool = False, step: int = 0) -> np.ndarray:
        """FP8-domain attention query scales by the same recipe: amax of the
        query (bf16 values) over the batch / 448, per tensor ([1]) or per q
        head ([Hq]); 1.0 where the amax is 0."""
        q = np.abs(bf16_bits_to_float(self.q(layer, step)))
        a = q.max(axis=(0, 2)) if per_head else np.array([q.max()])
        return np.where(a > 0, a / np.float32(448.0), 1.0).astype(np.float32)

    def scales(self, layer: int = 0) -> np.ndarray:
        """float32 [2]: FP8 {k_scale, v_scale} or NVFP4 {g_k, g_v} = amax / format max,
        amax taken over every generated K (resp. V) value of the layer; 1.0 otherwise
        (and in the default-scale mode)."""
        if layer not in self._scales:
            self.kv_all(layer)
        return self._scales[layer]


def make_page_table(seq_lens, P: int, seed: int, slack_pages: int = 0, max_pages: int | None = None):
    """Random page permutation: returns (page_table int32 [B][max_pages], num_pages)."""
    seq_lens = np.asarray(seq_lens, np.int64)
    npages = (seq_lens + P - 1) // P
    num_pages = int(npages.sum()) + slack_pages
    mp = int(npages.max()) if max_pages is None else max_pages
    mp = max(mp, 1)
    g = _gen(seed, 4)
    perm = torch.randperm(max(num_pages, 1), generator=g).numpy().astype(np.int32)
    pt = np.full((len(seq_lens), mp), -1, np.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt, max(num_pages, 1)


def make_workload(name: str, fmt: str, *, layers=1, Hq=64, Hkv=8, D=128, P=16, seq_lens=None,
                  B=1, T=None, T_range=None, seed=1000, k_outliers=(8, 10.0, 30.0), v_std=0.5,
                  v_token_sigma=0.5, scale_mode="amax", slack_pages=0) -> Workload:
    if seq_lens is None:
        if T_range is not None:
            g = _gen(seed, 5)
            lo, hi = T_range
            seq_lens = torch.randint(lo, hi + 1, (B,), generator=g).numpy()
        else:
            seq_lens = np.full(B, T)
    seq_lens = np.asarray(seq_lens, np.int32)
    pt, num_pages = make_page_table(seq_lens, P, seed, slack_pages)
    nc, lo, hi = k_outliers
    return Workload(name=name, fmt=fmt, layers=layers, Hq=Hq, Hkv=Hkv, D=D, P=P,
                    seq_lens=seq_lens, page_table=pt, num_pages=num_pages, seed=seed,
                    k_outlier_channels=nc, k_outlier_lo=lo, k_outlier_hi=hi, v_std=v_std,
                    v_token_sigma=v_token_sigma, scale_mode=scale_mode)


# ---- the workloads the library is specified on ------------------------------

def cfg1_e4m3_small(seed=1001) -> Workload:
    """Single layer, E4M3fn: Hq 32, Hkv 8, d 128, batch 2, context 256, random pages;
    Q, K, V ~ N(0, 1); K has 4 outlier channels per kv head scaled x20."""
    return make_workload("cfg1_e4m3_small", "fp8_e4m3", Hq=32, Hkv=8, B=2, T=256, seed=seed,
                         k_outliers=(4, 20.0, 20.0), v_std=1.0, v_token_sigma=0.0)


def cfg2_llama8b_stack(fmt="fp8_e5m2", seed=1002, layers=32, scale_mode="amax") -> Workload:
    """Llama-3-8B-shaped stack: 32 layers, Hq 32, Hkv 8; batch 8, lengths U[1K, 4K];
    K outliers 8 channels x U[10, 30]; V ~ N(0, 0.5^2) x lognormal(0, 0.5) per token."""
    return make_workload(f"cfg2_llama8b_stack_{fmt}", fmt, layers=layers, Hq=32, Hkv=8, B=8,
                         T_range=(1024, 4096), seed=seed, scale_mode=scale_mode)


def cfg3_fp4b16_70b(seed=1003) -> Workload:
    """FP4 block-16 (E8M0) on a 70B layer: Hq 64, Hkv 8; batch 8 at 16K."""
    return make_workload("cfg3_fp4b16_70b_16k", "fp4_mx_block16", Hq=64, Hkv=8, B=8, T=16384,
                         seed=seed)


def cfg4_nvfp4_70b_32k(seed=1004, B=32) -> Workload:
    """NVFP4 on a 70B layer: batch 32, ragged lengths U[24K, 32K], random page tables,
    g = amax / (448 * 6) per tensor.  (B < 32 only for profiling captures.)"""
    return make_workload("cfg4_nvfp4_70b_32k", "nvfp4", Hq=64, Hkv=8, B=B,
                         T_range=(24576, 32768), seed=seed)


def cfg5_sweep_cell(fmt: str, T: int, B: int, seed=1005) -> Workload:
    """One cell of the format sweep on a 70B layer (T in {4K, 16K, 32K}, B in {1, 8, 32})."""
    return make_workload(f"cfg5_{fmt}_{T // 1024}k_x{B}", fmt, Hq=64, Hkv=8, B=B, T=T, seed=seed)
