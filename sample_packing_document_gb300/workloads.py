"""Seeded synthetic inputs: document lengths, token ids, Q / K / V / dO.

This module draws random numbers and nothing else: it holds none of the
packing or attention arithmetic, so the CUDA path and the CPU oracle can both
take their inputs from it without sharing any of the method.

Workloads (document-length mixes and attention shapes of the five cases the
library is measured on; all data synthetic, no dataset is needed):

  tiny    one 256-token row (packed, micro_bsz 2, SEQ_LEN 128); document
          lengths uniform in [1, 64]; 2 heads, head_dim 64.
  c2      4 rows of 8192 (micro_bsz 2, SEQ_LEN 4096); lengths lognormal with
          median 600 and sigma 1.0, rounded, clipped to [16, 8192];
          32 q heads = 32 kv heads, head_dim 128.
  c3      one packed row of 32768 (micro_bsz 4, SEQ_LEN 8192); lengths 70%
          uniform [32, 1024], 30% uniform [4096, 16384]; GQA 32 q / 8 kv heads,
          head_dim 128, q drawn as N(0, 1) / sqrt(128). Also packed with
          use_packed_dataset=False (micro_bsz 4, SEQ_LEN 8192).
  c4      131072 tokens (micro_bsz 1, SEQ_LEN 131072); power-law lengths
          p(L) ~ L^-1.5 on [64, 65536] by inverse CDF, floored; 7 q heads /
          1 kv head (one rank's share of 56 / 8 heads over 8 sequence-parallel
          ranks), head_dim 128.
  c5      1,048,576 tokens (micro_bsz 1, SEQ_LEN 1048576); lengths 95% uniform
          [16, 512], 5% uniform [32768, 131072]; 4 q / 4 kv heads, head_dim 128.

Documents are drawn until their total reaches the target; the last one is cut
so the total is exactly the target (no padding in these cases). Token ids are
uniform in [1, 50000). Lengths and ids use numpy default_rng(seed) with
seed = case index; Q / K / V / dO are fp32 N(0, 1) from a torch generator
seeded with 100 + seed, rounded to bf16.
"""
import dataclasses

import numpy as np

VOCAB_LO, VOCAB_HI = 1, 50000


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    micro_bsz: int
    seq_len: int
    use_packed_dataset: bool
    target_tokens: int
    Hq: int
    Hkv: int
    head_dim: int
    q_scale: float = 1.0
    docs: str = ""        # name of the workload whose documents these are (default: this one)

    @property
    def docs_name(self):
        return self.docs or self.name


WORKLOADS = {
    "tiny": Workload("tiny", 0, 2, 128, True, 256, 2, 2, 64),
    "c2": Workload("c2", 1, 2, 4096, True, 32768, 32, 32, 128),
    "c3": Workload("c3", 2, 4, 8192, True, 32768, 32, 8, 128, q_scale=1.0 / np.sqrt(128.0)),
    "c3_unpack": Workload("c3_unpack", 2, 4, 8192, False, 32768, 32, 8, 128,
                          q_scale=1.0 / np.sqrt(128.0)),
    "c4": Workload("c4", 3, 1, 131072, True, 131072, 7, 1, 128),
    "c5": Workload("c5", 4, 1, 1048576, True, 1048576, 4, 4, 128),
    # c2's documents with 16 / 16 heads: a smaller device footprint for
    # hardware-counter captures (inputs still larger than L2).
    "c2p": Workload("c2p", 1, 2, 4096, True, 32768, 16, 16, 128, docs="c2"),
    # c5's documents with one q / kv head: the million-token row within a few GB
    # of device memory for hardware-counter captures.
    "c5p": Workload("c5p", 4, 1, 1048576, True, 1048576, 1, 1, 128, docs="c5"),
}


def _draw_length(name, rng):
    if name == "tiny":
        return int(rng.integers(1, 65))
    if name in ("c2", "c2p"):
        return int(np.clip(np.rint(np.exp(rng.normal(np.log(600.0), 1.0))), 16, 8192))
    if name.startswith("c3"):
        if rng.random() < 0.7:
            return int(rng.integers(32, 1025))
        return int(rng.integers(4096, 16385))
    if name == "c4":
        a, b, alpha = 64.0, 65536.0, 1.5
        u = rng.random()
        ea, eb = a ** (1 - alpha), b ** (1 - alpha)
        return int(np.floor((ea - u * (ea - eb)) ** (1.0 / (1 - alpha))))
    if name in ("c5", "c5p"):
        if rng.random() < 0.95:
            return int(rng.integers(16, 513))
        return int(rng.integers(32768, 131073))
    raise KeyError(name)


def doc_lengths(w: Workload):
    """Document lengths summing exactly to w.target_tokens."""
    rng = np.random.default_rng(w.seed)
    lens, total = [], 0
    while total < w.target_tokens:
        n = _draw_length(w.name, rng)
        n = min(n, w.target_tokens - total)
        lens.append(n)
        total += n
    return np.asarray(lens, dtype=np.int32)


def tokens(w: Workload, n_tokens):
    rng = np.random.default_rng(1000 + w.seed)
    return rng.integers(VOCAB_LO, VOCAB_HI, size=n_tokens, dtype=np.int64).astype(np.int32)


def documents(w: Workload):
    """(doc_lens int32 [num_docs], concatenated token ids int32 [num_tokens])."""
    lens = doc_lengths(w)
    return lens, tokens(w, int(lens.sum()))


def random_docs(rng, n_docs, len_lo, len_hi):
    """Small ad-hoc cases: n_docs documents with lengths uniform in
    [len_lo, len_hi]. Returns (doc_lens, tokens) as int32 arrays."""
    lens = rng.integers(len_lo, len_hi + 1, size=n_docs).astype(np.int32)
    toks = rng.integers(VOCAB_LO, VOCAB_HI, size=int(lens.sum())).astype(np.int32)
    return lens, toks


def qkv(T, Hq, Hkv, d, seed, device="cpu", q_scale=1.0):
    """bf16 q [T, Hq, d], k [T, Hkv, d], v [T, Hkv, d], dout [T, Hq, d]."""
    import torch
    g = torch.Generator(device=device).manual_seed(100 + seed)

    def draw(H, s=1.0):
        x = torch.randn(T, H, d, generator=g, device=device, dtype=torch.float32)
        if s != 1.0:
            x.mul_(s)
        return x.to(torch.bfloat16)

    q = draw(Hq, q_scale)
    k = draw(Hkv)
    v = draw(Hkv)
    do = draw(Hq)
    return q, k, v, do
