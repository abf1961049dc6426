"""Model shapes and the synthetic workloads they are measured on.

The drafter is a small pre-norm decoder stack (RMSNorm, GQA attention with
per-head q/k RMSNorm and rotate-half RoPE, SwiGLU MLP).  Its context comes
from hidden states tapped at several layers of a target model, fused by a
linear layer into one feature, and injected as K/V into every draft layer
(DFlash: how block diffusion boosts NVIDIA Blackwell throughput, section
"Block diffusion architecture").
"""
from dataclasses import dataclass, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    mlp: int
    vocab: int
    rms_eps: float = 1e-6
    rope_base: float = 1e6
    qk_norm: bool = True
    # K/V cache terms on the GPU: 2 = bf16 hi + lo planes (the target caches,
    # whose 8-layer logits need it to stay within 0.05 of exact arithmetic)
    kv_terms: int = 1

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def qkv_rows(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    def layer_params(self) -> int:
        h = self.hidden
        return (self.qkv_rows * h + h * self.q_dim + 3 * self.mlp * h
                + 2 * h + 2 * self.head_dim)


@dataclass(frozen=True)
class DraftShape(ModelShape):
    block: int = 16                 # anchor + (block - 1) mask positions
    n_taps: int = 5                 # target layers fused into the context feature
    conv_width: int = 0             # DFlash-2 depthwise block conv width (0 = off)
    fc_norm: bool = True            # RMSNorm after the fuse linear

    def params(self) -> int:
        h = self.hidden
        fuse = h * self.n_taps * h + h
        conv = self.n_layers * h * self.conv_width
        return fuse + self.n_layers * self.layer_params() + conv + 2 * h


@dataclass(frozen=True)
class Workload:
    """One measured configuration.

    ``ctx_len`` is the draft context length before this step's new context
    rows are appended; ``new_rows`` the rows appended per request in the
    step (``None`` = drawn per request as n_b + 1 of a previous verify).
    """
    wid: int
    name: str
    draft: DraftShape
    batch: int
    ctx_len: Optional[int] = None          # fixed length, or None = drawn
    ctx_len_range: Tuple[int, int] = (0, 0)
    new_rows: Optional[int] = 16
    agree_p: Optional[float] = 0.85        # fixed p, or None = drawn per request
    agree_p_range: Tuple[float, float] = (0.0, 0.0)
    page_size: int = 16
    shuffle_pages: bool = True
    target: Optional[ModelShape] = None
    tap_layers: Tuple[int, ...] = ()
    prompt_len: int = 0
    gen_tokens: int = 0
    description: str = ""


QWEN3_8B_DRAFT = DraftShape(n_layers=5, hidden=4096, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, mlp=12288, vocab=151936,
                            rms_eps=1e-6, rope_base=1e6, block=16, n_taps=5)

DFLASH2_DRAFT = DraftShape(n_layers=8, hidden=2048, n_q_heads=16, n_kv_heads=4,
                           head_dim=128, mlp=6144, vocab=151936,
                           rms_eps=1e-6, rope_base=1e6, block=16, n_taps=5,
                           conv_width=3)

TINY_TARGET = ModelShape(n_layers=4, hidden=256, n_q_heads=4, n_kv_heads=4,
                         head_dim=64, mlp=768, vocab=1024, rms_eps=1e-6,
                         rope_base=1e4, kv_terms=2)
TINY_DRAFT = DraftShape(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=4,
                        head_dim=64, mlp=768, vocab=1024, rms_eps=1e-6,
                        rope_base=1e4, block=8, n_taps=3)

E2E_TARGET = ModelShape(n_layers=8, hidden=4096, n_q_heads=32, n_kv_heads=8,
                        head_dim=128, mlp=12288, vocab=151936, rms_eps=1e-6,
                        rope_base=1e6, kv_terms=2)

WORKLOADS = {
    "tiny_e2e": Workload(
        wid=1, name="tiny_e2e", draft=TINY_DRAFT, batch=1, target=TINY_TARGET,
        tap_layers=(1, 2, 3), prompt_len=64, gen_tokens=128, ctx_len=None,
        new_rows=None, agree_p=None,
        description="4-layer H=256 target, 2-layer B=8 drafter, prompt 64, "
                    "generate 128, greedy"),
    "qwen3_8b_b1": Workload(
        wid=2, name="qwen3_8b_b1", draft=QWEN3_8B_DRAFT, batch=1, ctx_len=2048,
        new_rows=16, agree_p=0.85,
        description="Qwen3-8B-shaped 5-layer drafter, batch 1, B=16, 2048-token "
                    "context + 16 appended rows, p=0.85"),
    "qwen3_8b_b32_paged": Workload(
        wid=3, name="qwen3_8b_b32_paged", draft=QWEN3_8B_DRAFT, batch=32,
        ctx_len=None, ctx_len_range=(1024, 8192), new_rows=None, agree_p=None,
        agree_p_range=(0.6, 0.95),
        description="same drafter, batch 32, paged context L~U[1024,8192], "
                    "ragged appends n_b+1"),
    "dflash2_b16": Workload(
        wid=4, name="dflash2_b16", draft=DFLASH2_DRAFT, batch=16, ctx_len=16384,
        new_rows=16, agree_p=0.85,
        description="DFlash-2-style 8-layer H=2048 drafter with width-3 block "
                    "conv, batch 16, 16384-token contexts"),
    "e2e_8layer": Workload(
        wid=5, name="e2e_8layer", draft=QWEN3_8B_DRAFT, batch=8,
        target=E2E_TARGET, tap_layers=(1, 2, 4, 6, 7), prompt_len=1024,
        gen_tokens=512, ctx_len=None, new_rows=None, agree_p=None,
        description="8-layer H=4096 target + 5-layer B=16 drafter, batch 8, "
                    "prompts 1024, generate 512"),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


def tiny_workload(name: str = "tiny_step", wid: int = 11, *, hidden=256,
                  n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=64, mlp=512,
                  vocab=1000, block=8, n_taps=3, conv_width=0, batch=2,
                  ctx_len=None, ctx_len_range=(40, 90), new_rows=None,
                  agree_p=None, agree_p_range=(0.5, 0.95), page_size=16,
                  rope_base=1e4, qk_norm=True, fc_norm=True) -> Workload:
    """A small drafter step the oracle finishes in well under a second."""
    d = DraftShape(n_layers=n_layers, hidden=hidden, n_q_heads=n_q_heads,
                   n_kv_heads=n_kv_heads, head_dim=head_dim, mlp=mlp,
                   vocab=vocab, rms_eps=1e-6, rope_base=rope_base,
                   qk_norm=qk_norm, block=block, n_taps=n_taps,
                   conv_width=conv_width, fc_norm=fc_norm)
    return Workload(wid=wid, name=name, draft=d, batch=batch, ctx_len=ctx_len,
                    ctx_len_range=ctx_len_range, new_rows=new_rows,
                    agree_p=agree_p, agree_p_range=agree_p_range,
                    page_size=page_size)


def with_changes(w: Workload, **kw) -> Workload:
    return replace(w, **kw)
