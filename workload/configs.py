"""The five synthetic workload shapes of the sparse-KV reuse step.

Shapes follow the workloads the AVSG page (arxivdaily 2609.37538, English
abstract: an 8K-entry buffer, multi-token prediction, long contexts) and the
Spin page (gist.science 2604.26837, section 2B: head-wise pages, 64 recency
buckets) describe.  Nothing here is a dataset item: every input is drawn by
the seeded generator in ``gen.c``.

A *unit* is one (request, kv-head); an *entry* is the KV row of one token, or
of one 16-token head-wise page when ``entry_tokens == 16``.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    requests: int
    kv_heads: int
    q_per_kv: int          # G: query heads sharing one kv-head
    context: int           # tokens per unit
    head_dim: int          # D: K row width (latent width when kv_shared)
    v_dim: int             # Dv
    entry_tokens: int      # 1 (token entries) or 16 (head-wise pages)
    kv_shared: bool        # V aliases K (latent cache)
    k: int                 # selected entries per unit per query token
    slots: int             # B: buffer slots per unit
    steps: int             # decode steps (MTP: iterations)
    tokens_per_step: int   # 1, or 3 for multi-token prediction
    p_keep: float          # keep probability from the previous step/iteration
    p_keep_token: float    # keep probability between tokens of one iteration
    zipf_frac: float       # share of fresh ids drawn Zipf over rank from the end
    zipf_s: float
    forced: str            # "edges": 0..3 and the last 32; "pages": {0, P-2, P-1}

    @property
    def units(self) -> int:
        return self.requests * self.kv_heads

    @property
    def num_entries(self) -> int:
        return self.context // self.entry_tokens

    @property
    def entry_k_bytes(self) -> int:
        return self.entry_tokens * self.head_dim * 2

    @property
    def entry_v_bytes(self) -> int:
        return 0 if self.kv_shared else self.entry_tokens * self.v_dim * 2

    @property
    def entry_bytes(self) -> int:
        return self.entry_k_bytes + self.entry_v_bytes

    @property
    def softmax_scale(self) -> float:
        return self.head_dim ** -0.5

    def forced_ids(self) -> list:
        n = self.num_entries
        if self.forced == "edges":
            ids = list(range(min(4, n))) + list(range(max(0, n - 32), n))
        elif self.forced == "pages":
            ids = [0, n - 2, n - 1]
        elif self.forced == "none":
            ids = []
        else:
            raise ValueError(self.forced)
        out, seen = [], set()
        for i in ids:
            if 0 <= i < n and i not in seen:
                seen.add(i)
                out.append(i)
        return out

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # 1 request x 1 kv-head, L=4096, k=256, B=1024, 32 steps, p_keep 0.8.
    "tiny": Workload("tiny", 1, 1, 1, 4096, 128, 128, 1, False, 256, 1024, 32, 1,
                     0.8, 0.8, 0.0, 1.1, "edges"),
    # 8 x 8 units, GQA 4, L=32768, k=2048, B=8192, 128 steps, p_keep 0.9,
    # 20% of fresh ids Zipf(1.1) over rank from the end.
    "batch": Workload("batch", 8, 8, 4, 32768, 128, 128, 1, False, 2048, 8192, 128, 1,
                      0.9, 0.9, 0.2, 1.1, "edges"),
    # 16 x 8 units, 3 query tokens per iteration, 0.85 within / 0.9 across.
    "mtp": Workload("mtp", 16, 8, 4, 65536, 128, 128, 1, False, 2048, 8192, 64, 3,
                    0.9, 0.85, 0.0, 1.1, "edges"),
    # 32 x 8 units, 16-token head-wise pages (8192 per unit), k=128 pages, B=512.
    "pages": Workload("pages", 32, 8, 4, 131072, 128, 128, 16, False, 128, 512, 128, 1,
                      0.9, 0.9, 0.0, 1.1, "pages"),
    # 4 requests x 1 kv-head shared by 16 q-heads, L=2^20, latent 576 (K=V),
    # k=2048, 256 steps; B swept over {2048, 4096, 8192, 16384}.
    "latent": Workload("latent", 4, 1, 16, 1 << 20, 576, 576, 1, True, 2048, 8192, 256, 1,
                       0.9, 0.9, 0.2, 1.1, "edges"),
}

LATENT_SLOT_SWEEP = (2048, 4096, 8192, 16384)


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.replace(**overrides) if overrides else w
