"""Seeded synthetic inputs for the workloads (no softmax arithmetic in here).

Shared by the benchmark, the smoke check and the tests, on both sides of a parity check: the
CUDA path and the oracle always receive the same tensor values (generated here, then copied to
the host for the oracle).  Shapes and distributions follow the workloads the pages measure
(Qwen-Image joint attention: 16,384 rows of 4,096 image + 256 text keys, "[WS1][kernels] Add
fixed-order joint-attention softmax for Qwen-Image", Benchmark), plus padded prompts, causal
rows with a sink, long bf16 / fp32 rows, and rows longer than a shared-memory stage.  No public
dataset is involved; every value is drawn from a seeded normal or uniform distribution.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: torch.dtype
    batch: int
    heads: int
    q_len: int
    key_len: int
    score_sigma: float
    seed: int
    causal: bool = False
    sink: bool = False
    pad: tuple[int, int, int] | None = None  # valid length = base + U{lo..hi} per batch entry
    dp_sigma: float = 1.0

    @property
    def rows(self) -> int:
        return self.batch * self.heads * self.q_len

    @property
    def esz(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()

    def describe(self) -> dict:
        return {"workload": self.name, "rows": self.rows, "key_len": self.key_len,
                "batch": self.batch, "heads": self.heads, "q_len": self.q_len,
                "dtype": str(self.dtype).replace("torch.", ""), "causal": self.causal,
                "sink": self.sink, "padding": self.pad, "scores": f"N(0,{self.score_sigma}^2)",
                "dP": f"N(0,{self.dp_sigma}^2)", "seed": self.seed}


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_fp32", torch.float32, 2, 4, 257, 257, 3.0, seed=0),
        Workload("qwen_image_bf16", torch.bfloat16, 1, 1, 16384, 4352, 4.0, seed=1),
        Workload("prompt_padding_bf16", torch.bfloat16, 4, 24, 1024, 4608, 4.0, seed=2,
                 pad=(4096, 32, 512)),
        Workload("sink_causal_bf16", torch.bfloat16, 2, 64, 2048, 2048, 3.0, seed=3,
                 causal=True, sink=True),
        Workload("large_bf16", torch.bfloat16, 1, 24, 8192, 8192, 5.0, seed=4),
        Workload("large_fp32", torch.float32, 1, 24, 8192, 8192, 5.0, seed=4),
        # rows longer than a shared-memory stage (262,144 keys): the streaming kernels
        Workload("long_rows_bf16", torch.bfloat16, 1, 8, 128, 262144, 4.0, seed=5),
    )
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, sigma: float, seed: int, dtype: torch.dtype, device) -> torch.Tensor:
    """sigma * N(0, 1) drawn in float32, rounded to ``dtype`` (nearest even)."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    return (x * sigma).to(dtype)


def valid_lengths(w: Workload) -> torch.Tensor | None:
    """int32 [batch] on the CPU: base + U{lo..hi} (inclusive), or None without padding."""
    if w.pad is None:
        return None
    base, lo, hi = w.pad
    u = torch.randint(lo, hi + 1, (w.batch,), generator=_gen("cpu", w.seed * 1000 + 4))
    return (base + u).to(torch.int32)


def sink_logits(w: Workload) -> torch.Tensor | None:
    """float32 [heads] on the CPU, N(0, 1), or None without a sink."""
    if not w.sink:
        return None
    return torch.randn(w.heads, generator=_gen("cpu", w.seed * 1000 + 3), dtype=torch.float32)


def scores(w: Workload, device, *, neg_inf_tail: bool = True, seed_offset: int = 0):
    """[rows, key_len] scores; with padding, keys past each batch entry's valid length are
    set to -inf (unless neg_inf_tail is False)."""
    x = normal((w.rows, w.key_len), w.score_sigma, w.seed * 1000 + 1 + 7919 * seed_offset,
               w.dtype, device)
    lens = valid_lengths(w)
    if lens is not None and neg_inf_tail:
        per_b = x.view(w.batch, w.heads * w.q_len, w.key_len)
        for b in range(w.batch):
            per_b[b, :, int(lens[b]):] = float("-inf")
    return x


def dprobs(w: Workload, device, *, seed_offset: int = 0):
    return normal((w.rows, w.key_len), w.dp_sigma, w.seed * 1000 + 2 + 7919 * seed_offset,
                  w.dtype, device)


def probs_like(w: Workload, device, *, seed_offset: int = 0):
    """A probability-shaped backward input that needs no softmax: u^4 * 5 / key_len with
    u ~ U(0, 1), so entries are >= 0 with mean 1 / key_len, rounded to the dtype."""
    u = torch.rand((w.rows, w.key_len), generator=_gen(device, w.seed * 1000 + 5 + 7919 * seed_offset),
                   device=device, dtype=torch.float32)
    return (u.pow(4) * (5.0 / w.key_len)).to(w.dtype)


def sample_rows(heads: int, q_len: int, key_len: int, sigma: float, seed: int, sample: int,
                dtype: torch.dtype, device) -> torch.Tensor:
    """One batch entry ([heads * q_len, key_len]) of seeded scores, the same for a given
    (seed, sample) wherever it is placed; used to re-embed rows at other batch positions."""
    return normal((heads * q_len, key_len), sigma, seed * 100003 + sample, dtype, device)


def mean_valid_keys(w: Workload) -> float:
    """Mean number of keys per row that can be valid under the workload's causal bound and
    valid lengths (the keys the kernels read)."""
    L, Sq = w.key_len, w.q_len
    v = float(L)
    if w.causal:
        v = L - Sq + (Sq + 1) / 2.0  # query i sees L - Sq + i + 1 keys
    lens = valid_lengths(w)
    if lens is not None:
        v = min(v, float(lens.double().mean()))
    return v


def algorithmic_bytes(w: Workload, *, valid_keys: float | None = None) -> dict:
    """Bytes the method must move per pass (valid-key reads, full-row writes, FP32 per-row
    outputs): fwd = esz*|V| + esz*L + 4, bwd = 2*esz*|V| + esz*L + 4 (+4 with a sink: the
    sink gradient re-reads LSE and delta, 8 bytes per row)."""
    L, esz, R = w.key_len, w.esz, w.rows
    v = float(L) if valid_keys is None else float(valid_keys)
    fwd = R * (esz * v + esz * L + 4)
    bwd = R * (2 * esz * v + esz * L + 4)
    sink = R * 8 if w.sink else 0
    return {"fwd": fwd, "bwd": bwd, "sink": sink, "total": fwd + bwd + sink}
