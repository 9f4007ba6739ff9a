"""The five seeded synthetic workloads of the DFlash draft + verify step.

Shapes follow the drafter descriptions on the DFlash pages (aisparkup.com/wiki/dflash,
"핵심 아이디어": multi-layer target features fused by a light projection, injected as
K/V into every drafter layer, a block of masked tokens drafted in one forward pass,
the target's LM head reused) sized like Qwen3-8B, Llama-3.1-8B and gpt-oss-120b
drafters.  Nothing here computes any part of the method: it only names sizes, seeds
and workload statistics.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    # drafter / target shapes
    d_model: int
    n_target_layers: int
    target_width: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    block_size: int
    # step shape
    batch: int
    ctx_len: int                 # T_b after this step's injection (fixed configs)
    ctx_range: tuple | None = None   # (lo, hi) inclusive: ragged T_b ~ U{lo..hi}
    dtype: str = "bf16"          # "bf16" or "f32"
    rope_theta: float = 1e6
    rms_eps: float = 1e-6
    logit_std: float = 2.0       # target verify logits ~ N(0, logit_std)
    agree_p: float = 0.8         # planted draft/target agreement per position
    temperature: float = 0.0     # 0 = greedy verification
    seed: int = 0
    mask_id: int = 0
    page_size: int = 16
    permute_pages: bool = False
    weight_std: float = 0.02
    gain_std: float = 0.02
    hidden_std: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def fuse_in(self) -> int:
        return self.n_target_layers * self.target_width

    @property
    def q_width(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def rows(self) -> int:
        return self.batch * self.block_size

    @property
    def max_ctx(self) -> int:
        return self.ctx_range[1] if self.ctx_range else self.ctx_len

    @property
    def max_pages(self) -> int:
        return -(-self.max_ctx // self.page_size)

    @property
    def max_position(self) -> int:
        return self.max_ctx + self.block_size

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload(
    name="tiny-f32", d_model=256, n_target_layers=3, target_width=256, n_layers=1,
    n_q_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=688, vocab=2048, block_size=4,
    batch=1, ctx_len=64, dtype="f32", rope_theta=1e6, logit_std=1.0, agree_p=0.7, seed=0)

QWEN3_8B_B1 = Workload(
    name="qwen3-8b-shaped-b1", d_model=4096, n_target_layers=5, target_width=4096,
    n_layers=5, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=12288, vocab=151936,
    block_size=16, batch=1, ctx_len=2048, rope_theta=1e6, logit_std=2.0, agree_p=0.8, seed=1)

QWEN3_8B_B32 = replace(
    QWEN3_8B_B1, name="qwen3-8b-shaped-b32-ragged", batch=32, ctx_len=4096,
    ctx_range=(512, 4096), agree_p=0.75, seed=2, permute_pages=True)

LLAMA31_8B_B8 = Workload(
    name="llama-3.1-8b-shaped-b8", d_model=4096, n_target_layers=5, target_width=4096,
    n_layers=5, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=14336, vocab=128256,
    block_size=16, batch=8, ctx_len=8192, rope_theta=5e5, logit_std=2.0, agree_p=0.7, seed=3)

GPT_OSS_120B_B64 = Workload(
    name="gpt-oss-120b-shaped-b64-t1", d_model=2880, n_target_layers=5, target_width=2880,
    n_layers=5, n_q_heads=64, n_kv_heads=8, head_dim=64, ffn_dim=2880, vocab=201088,
    block_size=16, batch=64, ctx_len=16384, rope_theta=1.5e5, logit_std=2.0, agree_p=0.6,
    temperature=1.0, seed=4)

ALL = [TINY, QWEN3_8B_B1, QWEN3_8B_B32, LLAMA31_8B_B8, GPT_OSS_120B_B64]
BY_NAME = {w.name: w for w in ALL}


def small_bf16(**kw) -> Workload:
    """A bf16 workload small enough for the oracle to finish in seconds while still
    spanning several GEMM tiles, several context pages and a ragged page tail."""
    base = Workload(
        name="small-bf16", d_model=512, n_target_layers=3, target_width=320, n_layers=2,
        n_q_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=704, vocab=3000, block_size=16,
        batch=2, ctx_len=200, ctx_range=(37, 200), rope_theta=1e6, logit_std=2.0,
        agree_p=0.75, seed=11, permute_pages=True)
    return replace(base, **kw)
