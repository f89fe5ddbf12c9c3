"""Workload shapes for per-step working-set recall.

Each entry describes one synthetic agent workspace: model attention shape
(layers, KV heads, query heads, head dim, RoPE base), the history length in
32-token logical blocks, the number of current-step queries and the execution
view budget (sink blocks + recent blocks + top-k).  The shapes follow the
workloads of "KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer
GPU" (§6: 32-token blocks, 256K to 10M-token workspaces, 32K/64K/80K views) on a
Qwen-27B-class attention shape.  Nothing here computes anything.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

BLOCK_TOKENS = 32  # KVMem §4.3: the implementation defaults to 32-token blocks


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    rope_theta: float
    kv_dtype: str          # "f32", "bf16" or "e4m3": K pages, raw K, V
    index_dtype: str       # Mean-K entries
    q_dtype: str           # RoPE-free current-step queries
    n_blocks: int          # complete historical blocks N
    n_queries: int         # current-step query tokens M_q
    sink_blocks: int       # S
    recent_blocks: int     # W
    view_blocks: int       # V_b = S + W + k
    planted_frac: float    # fraction of non-reserved blocks with planted affinity
    n_planted: int = 0     # exact count (overrides planted_frac when > 0)
    k_shift: float = 2.0   # planted shift along u, in units of the K std
    q_shift: float = 1.5   # query shift along u
    k_std: float = 1.0     # std of raw K / V entries
    repo: str = "device"   # where raw K / V of the history live: device | host
    index_loc: str = "device"  # where the Mean-K index lives: device | host
    tile_blocks: int = 1024    # index tile for host-resident scoring
    steps: int = 1             # consecutive agent steps (churn workload)
    append_blocks: int = 0     # blocks appended to the history per step
    overlap: float = 0.0       # planted-topic overlap between consecutive steps
    n_topics: int = 1          # planted topic directions
    topics_per_step: int = 1

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def topk(self) -> int:
        return self.view_blocks - self.sink_blocks - self.recent_blocks

    @property
    def n_tokens(self) -> int:
        return self.n_blocks * BLOCK_TOKENS

    @property
    def view_tokens(self) -> int:
        return self.view_blocks * BLOCK_TOKENS

    def elem_bytes(self, which: str) -> int:
        return {"f32": 4, "bf16": 2, "e4m3": 1}[getattr(self, which)]

    @property
    def block_bytes(self) -> int:
        """Bytes of one block's K (or V) across all layers and KV heads."""
        return (self.n_layers * self.n_kv_heads * BLOCK_TOKENS * self.head_dim
                * self.elem_bytes("kv_dtype"))

    @property
    def index_entry_bytes(self) -> int:
        """Mean-K bytes of one block across all layers and KV heads."""
        return self.n_layers * self.n_kv_heads * self.head_dim * self.elem_bytes("index_dtype")

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Tiny correctness workspace: fp32, 128 blocks, 6 needle blocks, 13-block view.
TINY = Workload(
    name="tiny-4k", n_layers=2, n_kv_heads=2, n_q_heads=4, head_dim=64, rope_theta=1e4,
    kv_dtype="f32", index_dtype="f32", q_dtype="f32", n_blocks=128, n_queries=16,
    sink_blocks=1, recent_blocks=4, view_blocks=13, planted_frac=0.0, n_planted=6,
    k_shift=2.0, q_shift=1.5, k_std=1.0)

# Qwen-27B-class attention shape (64 layers, 8 KV heads, 48 query heads, d=128).
_Q27 = dict(n_layers=64, n_kv_heads=8, n_q_heads=48, head_dim=128, rope_theta=1e6,
            kv_dtype="bf16", index_dtype="bf16", q_dtype="bf16", n_queries=32,
            sink_blocks=4, recent_blocks=32, k_std=1.0 / 128 ** 0.5)

# One step at a 256K-token workspace, everything resident in HBM, 32K-token view.
W256K = Workload(name="q27-256k", n_blocks=8192, view_blocks=1024, planted_frac=0.02, **_Q27)

# 1M-token workspace on a 16-layer slice: raw K/V and the Mean-K index in pinned
# host memory, index scored in 1024-block tiles, 80K-token view.
W1M = Workload(name="q27x16-1m", n_blocks=32768, view_blocks=2560, planted_frac=0.02,
               repo="host", index_loc="host", tile_blocks=1024,
               **{**_Q27, "n_layers": 16})

# 20 agent steps over a 512K-token history, 64K-token view, 2048 tokens appended per
# step, planted-affinity blocks overlapping 70% between consecutive steps.
CHURN512K = Workload(name="q27-512k-churn", n_blocks=16384, view_blocks=2048,
                     planted_frac=0.02, repo="host", steps=20, append_blocks=64,
                     overlap=0.7, n_topics=64, topics_per_step=10, **_Q27)

# Scoring-only scaling point: a 10M-token Mean-K index (312500 blocks) in HBM.
W10M = Workload(name="q27-10m-score", n_blocks=312500, view_blocks=2048,
                planted_frac=0.005, **_Q27)

# The churn workload on a 16-layer slice: its 64-layer raw K / V (148 GB) does
# not fit pinned in the 199 GB of host memory next to the rest of the process.
CHURN512K_16 = CHURN512K.with_(name="q27x16-512k-churn", n_layers=16)

# The 256K step with 8-bit (e4m3) K / V pages, as the FP8 KV cache of the
# pages' evaluation platforms ([KVMem] §6.1); the index and queries stay bf16.
W256K_FP8 = W256K.with_(name="q27-256k-fp8", kv_dtype="e4m3")

ALL = {w.name: w for w in (TINY, W256K, W1M, CHURN512K, CHURN512K_16, W10M, W256K_FP8)}
