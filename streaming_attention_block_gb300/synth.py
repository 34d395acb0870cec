"""Seeded synthetic inputs for streaming chunk attention.

This module only draws numbers: it holds none of the attention, ring or
quantisation arithmetic, so the parity tests may feed the same tensors to the
CUDA library and to the CPU oracle.

Workloads (shapes from the pages, values synthetic: no page publishes data):

* ``tiny``: B=1, H=2, D=64, 32 tokens per chunk, ring of 2 cached chunks,
  window = current + 2 previous, 6 chunks, current chunk passed in.
* ``wan13b``: the Wan-1.3B streaming shape of "WanToFight" (30 DiT blocks, 4
  denoise steps, rolling cache of 2 chunks): B=1, H=12, D=128, 1536 tokens per
  chunk (2 latent frames x 24 x 32 patches), 20 chunks x 4 steps x 30 layers;
  Q and K RMS-normalised per token over H*D before rounding to bf16.
* ``long_sink``: the Matrix-Game 4.0 window shape (405 tokens per chunk, a
  reference chunk plus the 20 most recent chunks): B=1, H=24, D=128, sink +
  20-slot ring, the current chunk written into its slot before attending,
  60 chunks (the ring wraps 3 times), KV split into 8 partitions.
* ``block_causal``: training / causal-adaptation shape, B=2, 20 x 1536 =
  30720 tokens, H=12, D=128, window 2.
* ``fp8_kv``: ``long_sink`` with an E4M3 KV cache; K/V drawn N(0,1) with 1% of
  entries multiplied by 8 (outliers).
* ``int8k_kv``: ``fp8_kv`` with INT8 keys and E4M3 values ("Matrix-Game 4.0",
  section "技术新颖性": INT8 keys, FP8 values per window interval).

All values are N(0,1) fp32 draws rounded to bf16.  Draw order for a stream:
for each chunk, for each denoise step, for each layer: Q, then K, then V.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    Lc: int                 # tokens per chunk
    R: int = 0              # ring slots (0: no ring, full-sequence mode)
    W: int = 2              # previous chunks attended
    chunks: int = 1
    steps: int = 1          # denoise steps per chunk
    layers: int = 1
    sink: bool = False
    kcur_separate: bool = True   # True: current chunk passed in; False: appended first
    splits: int = 1
    kv_fp8: bool = False          # 8-bit cache (E4M3 keys and values, or INT8 keys with kv_int8k)
    kv_int8k: bool = False
    rms_norm: bool = False
    outliers: bool = False
    seq_chunks: int = 0     # full-sequence mode: chunks per sequence
    mem_pad: int = 0        # full-sequence mode: memory positions ahead of the target chunks
    mem_lens: tuple = ()    # real memory positions per sample (the rest is padding)
    seed: int = 1000

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=2, D=64, Lc=32, R=2, W=2, chunks=6, seed=1001),
    "wan13b": Workload("wan13b", B=1, H=12, D=128, Lc=1536, R=2, W=2, chunks=20, steps=4,
                       layers=30, rms_norm=True, seed=1002),
    "long_sink": Workload("long_sink", B=1, H=24, D=128, Lc=405, R=20, W=19, chunks=60,
                          sink=True, kcur_separate=False, splits=8, seed=1003),
    "block_causal": Workload("block_causal", B=2, H=12, D=128, Lc=1536, W=2, seq_chunks=20,
                             seed=1004),
    # compressed-memory training: 4 target chunks behind a padded memory of
    # two chunks' length, one sample's memory full and one's partly padding
    "memory_prefix": Workload("memory_prefix", B=2, H=12, D=128, Lc=1536, W=3, seq_chunks=4, mem_pad=3072,
                              mem_lens=(3072, 1900), seed=1007),
    "fp8_kv": Workload("fp8_kv", B=1, H=24, D=128, Lc=405, R=20, W=19, chunks=60, sink=True,
                       kcur_separate=False, splits=8, kv_fp8=True, outliers=True, seed=1005),
    "int8k_kv": Workload("int8k_kv", B=1, H=24, D=128, Lc=405, R=20, W=19, chunks=60, sink=True,
                         kcur_separate=False, splits=8, kv_fp8=True, kv_int8k=True, outliers=True, seed=1006),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def generator(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(gen: torch.Generator, shape, device: str = "cpu", rms_norm: bool = False,
               outliers: bool = False) -> torch.Tensor:
    """N(0,1) fp32 draw -> optional shaping -> bf16.

    ``rms_norm``: divide each token (last two dims H*D of a ``[B, L, H, D]``
    draw) by sqrt(mean(x^2) + 1e-6) in fp32 before rounding.
    ``outliers``: multiply 1% of entries (Bernoulli draw after the normal
    draw) by 8.
    """
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32, device=device)
    if outliers:
        sel = torch.rand(tuple(shape), generator=gen, dtype=torch.float32, device=device) < 0.01
        x = torch.where(sel, x * 8.0, x)
    if rms_norm:
        ms = x.pow(2).flatten(-2).mean(-1, keepdim=True).unsqueeze(-1)
        x = x / torch.sqrt(ms + 1e-6)
    return x.to(torch.bfloat16)


def chunk_qkv(w: Workload, gen: torch.Generator, device: str = "cpu"):
    """One (chunk, step, layer) draw: Q, K, V token-major ``[B, Lc, H, D]`` bf16."""
    shape = (w.B, w.Lc, w.H, w.D)
    q = randn_bf16(gen, shape, device, rms_norm=w.rms_norm)
    k = randn_bf16(gen, shape, device, rms_norm=w.rms_norm, outliers=w.outliers)
    v = randn_bf16(gen, shape, device, outliers=w.outliers)
    return q, k, v


def sink_kv(w: Workload, gen: torch.Generator, device: str = "cpu"):
    """Sink / reference chunk K, V token-major ``[B, Lc, H, D]`` bf16."""
    shape = (w.B, w.Lc, w.H, w.D)
    return (randn_bf16(gen, shape, device, outliers=w.outliers),
            randn_bf16(gen, shape, device, outliers=w.outliers))


def full_sequence_qkv(w: Workload, gen: torch.Generator, device: str = "cpu", seq_chunks: int | None = None):
    """Full-sequence Q, K, V ``[B, L, H, D]`` bf16 with L = mem_pad + seq_chunks * Lc."""
    n = w.seq_chunks if seq_chunks is None else seq_chunks
    shape = (w.B, w.mem_pad + n * w.Lc, w.H, w.D)
    return tuple(randn_bf16(gen, shape, device) for _ in range(3))
