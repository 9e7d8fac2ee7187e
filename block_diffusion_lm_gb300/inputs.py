"""Seeded synthetic inputs for block-diffusion attention workloads.

This module holds workload shapes and random number generation only: no step
of the attention method.  Both the CUDA path's tests/benchmark and the CPU
oracle's checks draw their inputs from here.

Every tensor is drawn as float32 N(0, 1) from one torch generator seeded with
`seed`, in the fixed order q_clean, k_clean, v_clean, q_corr, k_corr, v_corr,
do_clean, do_corr, then rounded to bfloat16 (round-to-nearest-even).  The
long fine-tune workload scales K of each KV head by s ~ U(0.5, 2) (drawn after
the tensors, before the bf16 rounding) to vary softmax sharpness.  Layout of
every tensor: [batch, L, heads, d] contiguous.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    L: int          # clean length = corrupted length
    M: int          # block size
    Hq: int
    Hkv: int
    d: int
    P: int = 1      # virtual clean shards (1 = unsharded fused path)
    has_clean_queries: bool = True
    k_scale_range: tuple | None = None   # per-KV-head K scale ~ U(lo, hi)
    seed: int = 1234
    window: int = 0                      # keys less than `window` positions back (0: all)
    clean_causal: bool = False           # clean queries token-causal (else block-causal)
    e4m3: bool = False                   # inputs kept in fp8 E4M3 (make_inputs_e4m3)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def B(self) -> int:
        return self.L // self.M

    def pairs_per_head(self) -> int:
        """Allowed (query, key) pairs per query head: L(L+M) with clean
        queries, L(L+M)/2 with corrupted queries only; with a window or
        token-causal clean queries, the sum of each row's key-range length."""
        if self.window <= 0 and not self.clean_causal:
            full = self.L * (self.L + self.M)
            return full if self.has_clean_queries else full // 2
        i = torch.arange(self.L, dtype=torch.int64)
        b = i // self.M
        lo = (i - self.window + 1).clamp(min=0) if self.window > 0 else torch.zeros_like(i)
        n = (b * self.M - lo).clamp(min=0)                                  # corrupted q, clean k
        n += ((b + 1) * self.M - torch.maximum(b * self.M, lo)).clamp(min=0)  # corrupted q, own block
        if self.has_clean_queries:
            hi = (i + 1) if self.clean_causal else (b + 1) * self.M
            n += (hi - lo).clamp(min=0)                                       # clean q, clean k
        return int(n.sum())

    def keys_of_row(self, q_stream: int, i: int) -> int:
        """Allowed keys of query row i of one copy (0 clean, 1 corrupted),
        counted the way pairs_per_head counts them."""
        b = i // self.M
        lo = max(0, i - self.window + 1) if self.window > 0 else 0
        if q_stream == 1:
            return max(0, b * self.M - lo) + max(0, (b + 1) * self.M - max(b * self.M, lo))
        hi = i + 1 if self.clean_causal else (b + 1) * self.M
        return max(0, hi - lo)

    def useful_fwd_flops(self) -> float:
        """QK^T and PV over allowed pairs: 4 d flops per pair per query head."""
        return 4.0 * self.d * self.pairs_per_head() * self.Hq * self.batch

    def useful_bwd_flops(self) -> float:
        """Backward at 2.5x forward (S recompute, dP, dV, dK, dQ)."""
        return 2.5 * self.useful_fwd_flops()


WORKLOADS = {
    # tiny MHA case the oracle finishes in seconds
    "tiny": Workload("tiny", 1, 1024, 64, 2, 2, 64, seed=1234),
    # dense 14B-like layer, GQA 40/8
    "dense14b": Workload("dense14b", 1, 16384, 32, 40, 8, 128, seed=1235),
    # context-sharded: P=8 virtual clean shards of 8192 tokens
    "sharded": Workload("sharded", 1, 65536, 64, 32, 8, 128, P=8, seed=1236),
    # long fine-tune layer, per-KV-head K scale, P=16
    "long": Workload("long", 1, 131072, 32, 32, 4, 128, P=16,
                     k_scale_range=(0.5, 2.0), seed=1237),
    # drafter: corrupted queries only over a 1M clean context
    "drafter": Workload("drafter", 1, 1048576, 16, 32, 8, 128,
                        has_clean_queries=False, seed=1238),
    # sliding-window layer: the dense shapes with a 1,024-token window
    "window1k": Workload("window1k", 1, 16384, 32, 40, 8, 128, window=1024, seed=1239),
    # the dense shapes with Q, K, V and dO kept in fp8 E4M3 (per-tensor scales)
    "dense14b_fp8": Workload("dense14b_fp8", 1, 16384, 32, 40, 8, 128, seed=1235, e4m3=True),
    # the dense shapes at the larger block sizes of the pages' training recipes
    "block128": Workload("block128", 1, 16384, 128, 40, 8, 128, seed=1240),
    "block256": Workload("block256", 1, 16384, 256, 40, 8, 128, seed=1241),
    "block512": Workload("block512", 1, 16384, 512, 40, 8, 128, seed=1242),
    "block1024": Workload("block1024", 1, 16384, 1024, 40, 8, 128, seed=1243),
}


def make_inputs(w: Workload, device="cuda", seed: int | None = None,
                L: int | None = None) -> dict:
    """Draw the workload's tensors on `device` (bf16, [batch, L, H, d]).

    `L` overrides the sequence length (same recipe, for scaled-down cases).
    """
    L = w.L if L is None else L
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)

    def draw(h):
        return torch.randn((w.batch, L, h, w.d), generator=g, device=device,
                           dtype=torch.float32)

    out = {}
    raw = {}
    for name, h in (("q_clean", w.Hq), ("k_clean", w.Hkv), ("v_clean", w.Hkv),
                    ("q_corr", w.Hq), ("k_corr", w.Hkv), ("v_corr", w.Hkv),
                    ("do_clean", w.Hq), ("do_corr", w.Hq)):
        if not w.has_clean_queries and name in ("q_clean", "do_clean"):
            continue
        raw[name] = draw(h)
    if w.k_scale_range is not None:
        lo, hi = w.k_scale_range
        s = lo + (hi - lo) * torch.rand((w.Hkv,), generator=g, device=device,
                                        dtype=torch.float32)
        raw["k_clean"] = raw["k_clean"] * s.view(1, 1, -1, 1)
        raw["k_corr"] = raw["k_corr"] * s.view(1, 1, -1, 1)
    for name, t in raw.items():
        out[name] = t.to(torch.bfloat16)
    if not w.has_clean_queries:
        out["q_clean"] = None
        out["do_clean"] = None
    return out


E4M3_MAX = 448.0  # largest finite E4M3 magnitude


def make_inputs_e4m3(w: Workload, device="cuda", seed: int | None = None,
                     L: int | None = None):
    """The workload's tensors drawn as in `make_inputs` (the same float32
    values before rounding), kept in fp8 E4M3: each tensor x gets a
    power-of-two scale s = 2^ceil(log2(max|x| / 448)) and is stored as the
    E4M3 rounding (nearest even) of x / s.  Returns ({name: uint8 tensor of
    the E4M3 codes}, {name: s}); names as in `make_inputs`, absent tensors
    None."""
    L = w.L if L is None else L
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    raw = {}
    for name, h in (("q_clean", w.Hq), ("k_clean", w.Hkv), ("v_clean", w.Hkv),
                    ("q_corr", w.Hq), ("k_corr", w.Hkv), ("v_corr", w.Hkv),
                    ("do_clean", w.Hq), ("do_corr", w.Hq)):
        if not w.has_clean_queries and name in ("q_clean", "do_clean"):
            continue
        raw[name] = torch.randn((w.batch, L, h, w.d), generator=g, device=device,
                                dtype=torch.float32)
    if w.k_scale_range is not None:
        lo, hi = w.k_scale_range
        s = lo + (hi - lo) * torch.rand((w.Hkv,), generator=g, device=device,
                                        dtype=torch.float32)
        raw["k_clean"] = raw["k_clean"] * s.view(1, 1, -1, 1)
        raw["k_corr"] = raw["k_corr"] * s.view(1, 1, -1, 1)
    codes, scales = {}, {}
    for name, t in raw.items():
        amax = float(t.abs().max().item())
        sc = 2.0 ** math.ceil(math.log2(amax / E4M3_MAX)) if amax > 0 else 1.0
        codes[name] = (t / sc).to(torch.float8_e4m3fn).view(torch.uint8)
        scales[name] = sc
    for name in ("q_clean", "do_clean"):
        if name not in codes:
            codes[name] = None
            scales[name] = None
    return codes, scales


def to_f64(t):
    """bf16 torch tensor (any device) -> float64 numpy array (exact up-cast)."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()


# ------------------------------------------------------------ vocabulary loss
@dataclasses.dataclass(frozen=True)
class CeWorkload:
    """LM-head cross-entropy: N loss rows of hidden size Dm against a V-row head."""
    name: str
    N: int
    Dm: int
    V: int
    chunk: int = 0            # rows per chunk (0: library default)
    head_grad: bool = True    # False: frozen head (no dW)
    ignore_frac: float = 0.0  # share of rows with target -1
    seed: int = 2000

    def flops(self) -> float:
        """Logits, dH and (trained head) dW: 2 N V Dm each."""
        return 2.0 * self.N * self.V * self.Dm * (3 if self.head_grad else 2)


CE_WORKLOADS = {
    "ce_tiny": CeWorkload("ce_tiny", 300, 192, 1600, chunk=128, ignore_frac=0.2, seed=2001),
    # LM head of the dense 14B-like layer: one 16K-token sequence, 128K vocabulary
    "lmhead14b": CeWorkload("lmhead14b", 16384, 5120, 131072, chunk=8192, seed=2002),
    # the drafter's frozen head (no dW)
    "lmhead_frozen": CeWorkload("lmhead_frozen", 16384, 5120, 131072, chunk=8192,
                                head_grad=False, seed=2003),
    # the same head on 2K rows: a case small enough for profiler captures
    # (logits chunk 256 MiB, still twice the L2)
    "lmhead_2k": CeWorkload("lmhead_2k", 2048, 5120, 32768, chunk=2048, seed=2004),
}


def make_ce_inputs(w: CeWorkload, device="cuda", seed: int | None = None) -> dict:
    """h ~ N(0, 1) [N, Dm] and W ~ N(0, 1) * 2/sqrt(Dm) [V, Dm] (logits of
    standard deviation about 2), both rounded to bf16; targets uniform over
    the vocabulary, a share `ignore_frac` of them set to -1.  Drawn from one
    torch generator in the order h, W, targets, ignore mask."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    h = torch.randn((w.N, w.Dm), generator=g, device=device, dtype=torch.float32)
    W = torch.randn((w.V, w.Dm), generator=g, device=device, dtype=torch.float32)
    W = W * (2.0 / math.sqrt(w.Dm))
    t = torch.randint(0, w.V, (w.N,), generator=g, device=device, dtype=torch.int64)
    drop = torch.rand((w.N,), generator=g, device=device) < w.ignore_frac
    t = torch.where(drop, torch.full_like(t, -1), t).to(torch.int32)
    n_valid = int((t >= 0).sum().item())
    return {"h": h.to(torch.bfloat16), "w": W.to(torch.bfloat16), "target": t,
            "grad_scale": 1.0 / max(1, n_valid)}
