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
    # seed of the per-sequence streams (context lengths, page order, target features,
    # verify logits, planting, uniforms); None = `seed`.  Weights always use `seed`, so
    # replicas that change only this share the drafter's weights.
    seq_seed: int | None = None
    mask_id: int = 0
    # projection weights: "native" (the dtype) or "fp8" (packed e4m3 with row scales)
    weight_format: str = "native"
    page_size: int = 16
    permute_pages: bool = False
    weight_std: float = 0.02
    gain_std: float = 0.02
    hidden_std: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def sseed(self) -> int:
        return self.seed if self.seq_seed is None else self.seq_seed

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


# Workloads the oracle finishes in seconds that still span several projection tiles,
# several context pages with a ragged last page, permuted pages and a ragged vocabulary
# tail; each exercises one launch configuration of the kernels (named in its comment).
PARITY_SMALL = {
    "tiny-f32": TINY,
    "small-bf16-hd128": small_bf16(),
    "small-bf16-hd64-g8": small_bf16(
        name="small-bf16-hd64-g8", d_model=384, n_q_heads=16, n_kv_heads=2, head_dim=64,
        ffn_dim=384, vocab=2176, batch=3, ctx_range=(16, 120), seed=12),
    # batch 1 x block 16 rows (the 16-row projection tiles), two and one context splits
    "small-bf16-b1": small_bf16(
        name="small-bf16-b1", batch=1, ctx_range=(150, 200), seed=14),
    "small-bf16-b1-1split": small_bf16(
        name="small-bf16-b1-1split", batch=1, ctx_range=(40, 100), seed=15),
    "small-bf16-b5-s8": small_bf16(
        name="small-bf16-b5-s8", block_size=8, batch=5, n_q_heads=4, n_kv_heads=2,
        ctx_range=(8, 70), vocab=1000, seed=13),
    # 96 and 320 block rows: the tcgen05 projection tiles (128 and 256 activation rows),
    # the second with a ragged 64-row second m-block; every tile split between CTAs
    "small-bf16-b6-tc128": small_bf16(
        name="small-bf16-b6-tc128", batch=6, ctx_range=(20, 90), seed=16),
    "small-bf16-b20-tc256": small_bf16(
        name="small-bf16-b20-tc256", batch=20, ctx_range=(16, 64), seed=17),
    # head_dim 64 with 96 and 80 block rows: attention on the tcgen05 kernel with 128 and
    # 64 query rows per kv head, ragged contexts over several splits and steps
    "small-bf16-hd64-g8-b6-tc": small_bf16(
        name="small-bf16-hd64-g8-b6-tc", d_model=384, n_q_heads=16, n_kv_heads=2,
        head_dim=64, ffn_dim=384, vocab=2176, batch=6, ctx_range=(16, 250), seed=19),
    "small-bf16-hd64-g4-b5-tc": small_bf16(
        name="small-bf16-hd64-g4-b5-tc", d_model=384, n_q_heads=8, n_kv_heads=2,
        head_dim=64, ffn_dim=384, vocab=2176, batch=5, ctx_range=(20, 180), seed=20),
    # one-page contexts (16 tokens: the split's single step holds the context page and
    # the block, so the tcgen05 key-split lanes of the step's second half see no valid
    # key) with 96 block rows at head_dim 128, and a mix of one- and two-page contexts
    # with 80 block rows at head_dim 64 (64 query rows per kv head)
    "small-bf16-b6-tc128-short": small_bf16(
        name="small-bf16-b6-tc128-short", batch=6, ctx_range=(16, 16), seed=22),
    "small-bf16-hd64-g4-b5-short": small_bf16(
        name="small-bf16-hd64-g4-b5-short", d_model=384, n_q_heads=8, n_kv_heads=2,
        head_dim=64, ffn_dim=384, vocab=2176, batch=5, ctx_range=(16, 24), seed=23),
    # 256 rows with K = 1024 and a 32000-token vocabulary: whole tiles per CTA as well
    "mid-bf16-b16-tc256": small_bf16(
        name="mid-bf16-b16-tc256", d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128,
        ffn_dim=2816, vocab=32000, batch=16, ctx_range=(16, 48), seed=18),
}


def one_layer(w: Workload) -> Workload:
    """The same shapes with a single drafter layer (fewer compounding rounding points)."""
    return replace(w, name=w.name + "-1l", n_layers=1)


ONE_LAYER = {v.name: v for v in (one_layer(QWEN3_8B_B1), one_layer(LLAMA31_8B_B8),
                                 one_layer(GPT_OSS_120B_B64))}


@dataclass(frozen=True)
class SpecWorkload:
    """The greedy speculative loop: a drafter (its target_width = d_model) and a random
    causal target transformer of the same width, heads, FFN and vocabulary with
    `target_layers` layers; the drafter fuses the target's outputs after `tap_layers`
    and reuses the target's embedding and LM head.  Every sequence starts from a
    `prompt_len`-token random prompt; `plant_p` is the per-position probability of the
    synthetic agreement that stands in for a trained drafter/target pair."""
    name: str
    drafter: Workload
    target_layers: int
    tap_layers: tuple
    prompt_len: int
    steps: int
    plant_p: float

    @property
    def target(self) -> Workload:
        return replace(self.drafter, name=self.name + "-target", n_layers=self.target_layers,
                       seed=self.drafter.seed + 104729)

    @property
    def max_position(self) -> int:
        # prompt, every step's block (up to S new tokens each) and one block of slack
        return self.prompt_len + (self.steps + 2) * self.drafter.block_size


SPEC_TINY = SpecWorkload(
    name="spec-tiny-f32", drafter=replace(TINY, name="spec-tiny-f32-drafter", batch=2),
    target_layers=4, tap_layers=(1, 2, 4), prompt_len=37, steps=6, plant_p=0.7)

SPEC_SMALL_BF16 = SpecWorkload(
    name="spec-small-bf16",
    drafter=small_bf16(name="spec-small-bf16-drafter", target_width=512, batch=3, seed=31),
    target_layers=4, tap_layers=(1, 2, 4), prompt_len=45, steps=6, plant_p=0.75)

# Qwen3-8B-shaped drafter (5 layers) against a 36-layer Qwen3-8B-shaped random target:
# five target layers spread over its depth are fused; agreement as in the batch-1 step
SPEC_QWEN3_8B = SpecWorkload(
    name="spec-qwen3-8b-shaped-b1", drafter=replace(QWEN3_8B_B1, name="spec-qwen3-8b-drafter"),
    target_layers=36, tap_layers=(4, 11, 18, 25, 32), prompt_len=2048, steps=64, plant_p=0.8)

SPEC = {s.name: s for s in (SPEC_TINY, SPEC_SMALL_BF16, SPEC_QWEN3_8B)}


def fp8(w: Workload, name=None) -> Workload:
    """The same workload with its projection weights streamed as FP8 (e4m3, per-row
    power-of-two scales)."""
    return replace(w, name=(name or w.name) + "-fp8", weight_format="fp8")


# FP8 weight streaming: 16-row blocks (batch 1), 32 rows (two blocks), 320 rows (many
# 32-row tiles of the weight-streaming kernel), and the Qwen3-8B-shaped batch-1 step
FP8 = {v.name: v for v in [fp8(PARITY_SMALL[k], k) for k in
                           ("small-bf16-b1", "small-bf16-hd128", "small-bf16-b20-tc256")]
       + [fp8(QWEN3_8B_B1)]}


def named(name: str) -> Workload:
    """Any workload defined here, by name (step workloads, parity workloads, one-layer
    and FP8 variants)."""
    for table in (BY_NAME, PARITY_SMALL, ONE_LAYER, FP8):
        if name in table:
            return table[name]
    raise KeyError(name)
