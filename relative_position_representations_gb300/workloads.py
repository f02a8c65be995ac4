"""Named workloads and the seeded synthetic-input generator.

This module holds shapes, distributions and random draws only: none of the attention
arithmetic. Both the CUDA path (through bench.py and the GPU tests) and the CPU oracle are
fed from here, so the two see bit-identical inputs.

Shapes follow the translation Transformer configurations on the "Self-Attention with
Relative Position Representations" page (section 5, "Evaluation Methodology": base d_z = 64
with 8 heads and clip k = 16, big d_z = 64 with 16 heads), plus a long-sequence key-only
case and the T5 bias case ("Relative position embeddings" page, section "T5": 32 buckets,
max_distance 128). No dataset is read:
every value is drawn from a torch CPU generator seeded by the caller.

Draw order (fp32 draws, then a round-to-nearest-even cast to the workload dtype):
Shaw: q, k, v, a^K, a^V, kv_len. T5: q, k, v, bias. Transformer-XL: q, k, v, rel, u, v, kv_len. ALiBi: q, k, v, kv_len (the slopes are
fixed, not drawn). Clipped offset table: q, k, v, table, kv_len. Labelled edges: q, k, v,
a^K, a^V (num_labels rows), labels ~ U{0..num_labels-1} per pair (uint8), kv_len. N(0, s^2) means s * randn.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dtype: str                      # "bf16" or "f32"
    kind: str = "shaw"              # "shaw", "t5", "alibi", "offset" (clipped per-offset scalar
                                    # table), "labeled" (label matrix), "txl" (Transformer-XL),
                                    # "decode" (one decoding step), "bwd" (gradients)
    clip_k: int = 0                 # Shaw clip distance; the table radius for "offset"
    causal: bool = False
    key_term: bool = True           # a^K present (Shaw)
    value_term: bool = True         # a^V present (Shaw)
    qkv_std: float = 1.0
    table_std: float = 0.02
    shared_tables: bool = False     # one table for all heads (head stride 0)
    kv_len_range: Optional[tuple] = None   # inclusive (lo, hi) per sequence, or None
    scale: Optional[float] = None   # default 1/sqrt(d) for Shaw, 1.0 for T5
    num_buckets: int = 32
    max_distance: int = 128
    bidirectional: bool = True
    bias_std: float = 1.0
    alibi_max_bias: float = 8.0     # ALiBi slopes m_h = 2^(-alibi_max_bias * (h + 1) / H)
    num_labels: int = 16            # "labeled": table rows (labels are uint8)
    labels_per_sequence: bool = True  # "labeled": one label matrix per sequence, else shared

    @property
    def softmax_scale(self) -> float:
        if self.scale is not None:
            return float(self.scale)
        return 1.0 if self.kind == "t5" else 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny fp32 case the oracle finishes instantly
    "tiny_fp32": Workload("tiny_fp32", B=1, H=2, n=16, d=8, dtype="f32", clip_k=2,
                          table_std=0.1, scale=1.0 / math.sqrt(8)),
    # Transformer-base encoder self-attention with per-sequence key padding
    "base_encoder": Workload("base_encoder", B=64, H=8, n=128, d=64, dtype="bf16", clip_k=16,
                             table_std=0.02, kv_len_range=(32, 128), scale=1.0 / 8),
    # Transformer-big decoder self-attention (causal)
    "big_decoder": Workload("big_decoder", B=32, H=16, n=256, d=64, dtype="bf16", clip_k=16,
                            table_std=0.02, causal=True, scale=1.0 / 8),
    # long sequence, key-relative term only, causal
    "long_keyonly": Workload("long_keyonly", B=4, H=16, n=4096, d=128, dtype="bf16",
                             clip_k=64, table_std=0.02, causal=True, value_term=False,
                             scale=1.0 / math.sqrt(128)),
    # T5 scalar bucketed bias, no 1/sqrt(d)
    "t5_bias": Workload("t5_bias", B=8, H=12, n=2048, d=64, dtype="bf16", kind="t5",
                        qkv_std=1.0 / 8, scale=1.0, num_buckets=32, max_distance=128,
                        bidirectional=True, bias_std=1.0),
}

ORDER = ["tiny_fp32", "base_encoder", "big_decoder", "long_keyonly", "t5_bias"]

# Scalar offset biases through the T5 form ("Relative position embeddings" page, sections
# "T5" and "Placement in the taxonomy"), on the T5 case's shape: ALiBi in a causal decoder
# (q, k, v ~ N(0, 1), 1/sqrt(d)), and a learned per-head scalar per offset clipped at 128
# (the T5 case's max_distance) in a bidirectional encoder.
BIAS_WORKLOADS = {
    "alibi_decoder": Workload("alibi_decoder", B=8, H=12, n=2048, d=64, dtype="bf16",
                              kind="alibi", causal=True, scale=1.0 / 8),
    "offset_bias": Workload("offset_bias", B=8, H=12, n=2048, d=64, dtype="bf16",
                            kind="offset", clip_k=128, scale=1.0 / 8, bias_std=1.0),
}

# Labelled edges ("Self-Attention with Relative Position Representations" page, section
# "Relation-Aware Self-Attention: The Core Modification"): a
# random graph with 16 edge types over 512 tokens per sequence, Transformer-base heads.
LABELED_WORKLOADS = {
    "labeled_graph": Workload("labeled_graph", B=16, H=8, n=512, d=64, dtype="bf16",
                              kind="labeled", num_labels=16, table_std=0.02, scale=1.0 / 8,
                              kv_len_range=(256, 512)),
}

# Transformer-XL ("Relative Position Encoding in Transformer-XL" page): a causal decoder of
# the T5 case's shape with projected encodings of every offset and the global biases u and v
# (all N(0, 0.5^2): large enough that every term moves the output).
TXL_WORKLOADS = {
    "txl_decoder": Workload("txl_decoder", B=8, H=12, n=1024, d=64, dtype="bf16", kind="txl",
                            causal=True, table_std=0.5, scale=1.0 / 8),
}

# Gradients (kind "bwd"): the forward's inputs plus dout ~ N(0, 1) drawn after them. The base
# encoder shape (one query tile per head) and the big decoder shape (two, causal).
BWD_WORKLOADS = {
    "bwd_base_encoder": Workload("bwd_base_encoder", B=64, H=8, n=128, d=64, dtype="bf16",
                                 kind="bwd", clip_k=16, table_std=0.02, kv_len_range=(32, 128),
                                 scale=1.0 / 8),
    "bwd_big_decoder": Workload("bwd_big_decoder", B=32, H=16, n=256, d=64, dtype="bf16",
                                kind="bwd", clip_k=16, table_std=0.02, causal=True,
                                scale=1.0 / 8),
}

# One incremental decoding step (kind "decode"): n is the cache capacity T; each sequence's
# cache holds kv_len_range-drawn entries, the last being the new token (Transformer-big
# decoder shape, caches of 1K-2K tokens).
DECODE_WORKLOADS = {
    "decode_big": Workload("decode_big", B=32, H=16, n=2048, d=64, dtype="bf16", kind="decode",
                           clip_k=16, causal=True, table_std=0.02, kv_len_range=(1024, 2048),
                           scale=1.0 / 8),
}


def draw_inputs(w: Workload, seed: int = 0) -> dict:
    """Seeded CPU tensors for workload w (see the module docstring for the recipe)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (w.B, w.H, w.n, w.d)
    dt = w.torch_dtype

    def normal(shp, std):
        return (torch.randn(shp, generator=g, dtype=torch.float32) * std).to(dt)

    out = {"q": normal(shape, w.qkv_std), "k": normal(shape, w.qkv_std),
           "v": normal(shape, w.qkv_std)}
    if w.kind == "t5":
        out["bias"] = torch.randn((w.num_buckets, w.H), generator=g,
                                  dtype=torch.float32) * w.bias_std
        out["kv_len"] = None
        return out
    if w.kind == "txl":  # projected offset encodings [H|1, 2n-1, d], then u and v [H|1, d]
        Ht = 1 if w.shared_tables else w.H
        out["rel"] = normal((Ht, 2 * w.n - 1, w.d), w.table_std)
        out["u"] = normal((Ht, w.d), w.table_std)
        out["vb"] = normal((Ht, w.d), w.table_std)
        out["kv_len"] = None
        if w.kv_len_range is not None:
            lo, hi = w.kv_len_range
            out["kv_len"] = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int32)
        return out
    if w.kind in ("alibi", "offset"):
        if w.kind == "alibi":
            out["slopes"] = alibi_slopes(w)
        else:
            Ht = 1 if w.shared_tables else w.H
            out["table"] = torch.randn((Ht, 2 * w.clip_k + 1), generator=g,
                                       dtype=torch.float32) * w.bias_std
        out["kv_len"] = None
        if w.kv_len_range is not None:
            lo, hi = w.kv_len_range
            out["kv_len"] = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int32)
        return out
    W = w.num_labels if w.kind == "labeled" else 2 * w.clip_k + 1
    Ht = 1 if w.shared_tables else w.H
    out["aK"] = normal((Ht, W, w.d), w.table_std) if w.key_term else None
    out["aV"] = normal((Ht, W, w.d), w.table_std) if w.value_term else None
    if w.kind == "labeled":
        shape_l = (w.B, w.n, w.n) if w.labels_per_sequence else (w.n, w.n)
        out["labels"] = torch.randint(0, w.num_labels, shape_l, generator=g,
                                      dtype=torch.int32).to(torch.uint8)
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        out["kv_len"] = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int32)
    else:
        out["kv_len"] = None
    return out


def draw_bwd_inputs(w: Workload, seed: int = 0) -> dict:
    """The forward inputs of a Shaw workload, then dout [B, H, n, d] ~ N(0, 1)."""
    x = draw_inputs(w.replace(kind="shaw"), seed)
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    x["dout"] = torch.randn((w.B, w.H, w.n, w.d), generator=g,
                            dtype=torch.float32).to(w.torch_dtype)
    return x


def draw_decode_inputs(w: Workload, seed: int = 0) -> dict:
    """Seeded CPU tensors for a decode step: q [B, H, d], k / v caches [B, H, T, d] with
    T = w.n, tables, and cache_len [B] int32 (draw order q, k, v, a^K, a^V, cache_len)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    dt = w.torch_dtype

    def normal(shp, std):
        return (torch.randn(shp, generator=g, dtype=torch.float32) * std).to(dt)

    out = {"q": normal((w.B, w.H, w.d), w.qkv_std),
           "k": normal((w.B, w.H, w.n, w.d), w.qkv_std),
           "v": normal((w.B, w.H, w.n, w.d), w.qkv_std)}
    W = 2 * w.clip_k + 1
    Ht = 1 if w.shared_tables else w.H
    out["aK"] = normal((Ht, W, w.d), w.table_std) if w.key_term else None
    out["aV"] = normal((Ht, W, w.d), w.table_std) if w.value_term else None
    lo, hi = w.kv_len_range if w.kv_len_range is not None else (w.n, w.n)
    out["cache_len"] = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int32)
    return out


def alibi_slopes(w: Workload) -> torch.Tensor:
    """The fixed ALiBi slopes, a geometric sequence over the heads: [H] fp32."""
    return torch.tensor([2.0 ** (-w.alibi_max_bias * (h + 1) / w.H) for h in range(w.H)],
                        dtype=torch.float32)


def table_head_stride(w: Workload) -> int:
    rows = w.num_labels if w.kind == "labeled" else 2 * w.clip_k + 1
    return 0 if w.shared_tables else rows * w.d
