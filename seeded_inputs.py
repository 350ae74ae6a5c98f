"""Seeded synthetic inputs and workload shapes for the attention-over-KV-cache path.

This module is the only code shared by the CPU oracle side (tests, cpu baseline)
and the GPU side (tests, bench).  It draws random numbers and describes the
workload shapes; it contains none of the method's arithmetic (no quantisation,
no attention, no serialisation).

Every tensor is drawn from its own stream (NumPy's SFC64 generator seeded by a
SeedSequence of (seed, layer, tensor id)), so a layer's Q, K and V never
depend on how many other layers or tensors were drawn.  The
prompt tokens and the decode tokens of one layer come from one stream: the
decode tokens are simply the rows after the prompt.

Values are N(0, 1) drawn in float32 and then rounded to the workload's input
dtype (round-to-nearest-even for bf16, via torch's CPU conversion).
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np
import torch

Q_ID, K_ID, V_ID, OUTLIER_ID = 0, 1, 2, 3


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: the shapes of the pages' runs, scaled to one layer.

    n_prompt tokens are prefilled in chunks of `chunk` tokens, then `n_decode`
    single-token decode steps follow.  `cache` is "q8_0" or "f16"; `in_dtype`
    is the dtype of Q/K/V as handed to the path ("f32" or "bf16").
    """

    name: str
    n_layer: int
    n_head_q: int
    n_head_kv: int
    head_dim: int
    cache: str
    in_dtype: str
    n_ctx: int
    n_prompt: int
    chunk: int
    n_decode: int
    seed: int
    k_outlier_frac: float = 0.0   # fraction of K channels scaled x4
    chunk_sweep: Tuple[int, ...] = ()

    @property
    def group(self) -> int:
        return self.n_head_q // self.n_head_kv

    @property
    def n_tokens(self) -> int:
        return self.n_prompt + self.n_decode

    def chunks(self, chunk: Optional[int] = None):
        """(pos0, length) of each prefill chunk of the prompt."""
        c = self.chunk if chunk is None else chunk
        if c <= 0:
            c = self.n_prompt
        return [(p, min(c, self.n_prompt - p)) for p in range(0, self.n_prompt, c)]


# The five workloads.  Sizes follow the pages' runs: a 256-token toy; the
# 17,055-token f16-cache request at context 20,480 in 512-token ubatches; the
# 58.3k-token q8_0 request at context 65,536 in 2048-token ubatches; the
# 10,041-token chunk-size sweep; and a 64-layer stack at 28,998 tokens.
WORKLOADS: Dict[str, Workload] = {
    "toy_q8_0": Workload("toy_q8_0", 1, 4, 2, 64, "q8_0", "f32",
                         n_ctx=512, n_prompt=256, chunk=64, n_decode=8, seed=1001),
    "f16_17k": Workload("f16_17k", 1, 40, 8, 128, "f16", "bf16",
                        n_ctx=20480, n_prompt=17055, chunk=512, n_decode=128, seed=1002),
    "q8_0_58k": Workload("q8_0_58k", 1, 40, 8, 128, "q8_0", "bf16",
                         n_ctx=65536, n_prompt=58300, chunk=2048, n_decode=256, seed=1003,
                         k_outlier_frac=0.01),
    "q8_0_sweep_10k": Workload("q8_0_sweep_10k", 1, 40, 8, 128, "q8_0", "bf16",
                               n_ctx=10240, n_prompt=10041, chunk=2048, n_decode=0, seed=1004,
                               chunk_sweep=(256, 512, 1024, 2048, 3328, 0)),
    "q8_0_stack64": Workload("q8_0_stack64", 64, 40, 8, 128, "q8_0", "bf16",
                             n_ctx=32768, n_prompt=28998, chunk=1024, n_decode=128, seed=1005),
}


def _stream(seed: int, layer: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, layer, tensor_id])))


def normal_rows(seed: int, layer: int, tensor_id: int, n_rows: int, n_head: int,
                head_dim: int) -> np.ndarray:
    """N(0,1) float32 rows [0, n_rows) of one tensor's stream, shape [n_rows, n_head, head_dim].

    Rows are drawn in order from the start of the stream, so a row's values do
    not depend on n_rows.
    """
    g = _stream(seed, layer, tensor_id)
    per_row = n_head * head_dim
    x = g.standard_normal(n_rows * per_row, dtype=np.float32)
    return x.reshape(n_rows, n_head, head_dim)


def outlier_channels(w: Workload, layer: int) -> np.ndarray:
    """Indices (into the flattened n_head_kv*head_dim channel axis) of K channels scaled x4."""
    n_ch = w.n_head_kv * w.head_dim
    n_out = int(round(w.k_outlier_frac * n_ch))
    if n_out == 0:
        return np.zeros(0, dtype=np.int64)
    g = _stream(w.seed, layer, OUTLIER_ID)
    return np.sort(g.choice(n_ch, size=n_out, replace=False)).astype(np.int64)


def to_input_dtype(x: np.ndarray, in_dtype: str) -> torch.Tensor:
    """Round float32 values to the workload's input dtype (RNE), as a CPU torch tensor."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if in_dtype == "f32":
        return t
    if in_dtype == "bf16":
        return t.to(torch.bfloat16)
    if in_dtype == "f16":
        return t.to(torch.float16)
    raise ValueError(in_dtype)


def layer_qkv(w: Workload, layer: int, n_rows: Optional[int] = None):
    """Q [n, H_q, D], K and V [n, H_kv, D] of one layer as CPU tensors in w.in_dtype.

    n defaults to prompt + decode tokens.  For workloads with K outliers, the
    seeded channel subset is multiplied by 4 before rounding to the input dtype.
    """
    n = w.n_tokens if n_rows is None else n_rows
    q = normal_rows(w.seed, layer, Q_ID, n, w.n_head_q, w.head_dim)
    k = normal_rows(w.seed, layer, K_ID, n, w.n_head_kv, w.head_dim)
    v = normal_rows(w.seed, layer, V_ID, n, w.n_head_kv, w.head_dim)
    ch = outlier_channels(w, layer)
    if ch.size:
        kf = k.reshape(n, -1)
        kf[:, ch] *= np.float32(4.0)
    return to_input_dtype(q, w.in_dtype), to_input_dtype(k, w.in_dtype), to_input_dtype(v, w.in_dtype)


def layer_qkv_device(w: Workload, layer: int, device, n_rows: Optional[int] = None):
    """Q, K, V of one layer drawn on a CUDA device (torch's counter-based Philox generator), in w.in_dtype.

    For large stacks where drawing on the host would take minutes.  The values
    differ from layer_qkv's (another generator) but are just as seeded: the
    same (seed, layer) always gives the same tensors, and a CPU copy of them is
    what the oracle receives.  K outliers follow the same seeded channel choice.
    """
    import hashlib
    n = w.n_tokens if n_rows is None else n_rows
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[w.in_dtype]
    out = []
    for tid, heads in ((Q_ID, w.n_head_q), (K_ID, w.n_head_kv), (V_ID, w.n_head_kv)):
        key = int.from_bytes(hashlib.sha256(b"%d/%d/%d" % (w.seed, layer, tid)).digest()[:8], "little") >> 1
        g = torch.Generator(device=device)
        g.manual_seed(key)
        x = torch.randn((n, heads, w.head_dim), generator=g, device=device, dtype=torch.float32)
        if tid == K_ID:
            ch = outlier_channels(w, layer)
            if ch.size:
                x.view(n, -1)[:, torch.from_numpy(ch).to(device)] *= 4.0
        out.append(x.to(dt))
    return tuple(out)


def small_workload(name: str, n_head_q: int, n_head_kv: int, head_dim: int, cache: str,
                   in_dtype: str, n_prompt: int, chunk: int, n_decode: int, seed: int,
                   n_ctx: Optional[int] = None, n_layer: int = 1,
                   k_outlier_frac: float = 0.0) -> Workload:
    """A reduced-size workload of the same structure, for parity tests the oracle finishes in seconds."""
    ctx = n_ctx if n_ctx is not None else n_prompt + n_decode + 16
    return Workload(name, n_layer, n_head_q, n_head_kv, head_dim, cache, in_dtype, ctx,
                    n_prompt, chunk, n_decode, seed, k_outlier_frac)


def sample_rows(seed: int, chunks, n_random: int = 6) -> np.ndarray:
    """Seeded query-row sample: each chunk's first and last row plus n_random rows per chunk."""
    g = np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, 99])))
    rows = []
    for p, c in chunks:
        rows += [p, p + c - 1]
        if c > 2:
            rows += list(p + 1 + g.choice(c - 2, size=min(n_random, c - 2), replace=False))
    return np.unique(np.asarray(rows, dtype=np.int64))
