"""Seeded synthetic inputs for the drafting-round tree builder.

This module only draws random tensors. It holds none of the builder's arithmetic (no top-M, no GRU, no scoring),
so the CUDA path and the CPU oracle can both read what it returns without sharing any method code.

The five workloads follow the shapes of a Qwen3-4B / Qwen3-8B drafting round: vocabulary V = 151936, block of
K = 16 positions, GRU hidden H and embedding width E of the drafter's correction, candidate width M, node budget n
(DominoTree summary on blog.captcha.la, "Key findings" and "Methodology — deep read"; gist.science explainer,
"Composants Clés"). No dataset or checkpoint is read: the marginal logits are Gaussian with a few strongly boosted
ids per position, which gives the peaked, long-tailed rows a block-diffusion drafter emits.

Recipe (every tensor has its own generator, so the draw order does not matter):
  * generator for tensor ``name``: ``torch.Generator(device).manual_seed(seed * 64 + STREAM[name])``,
    ``seed = 1234 + 100 * config`` by default;
  * logits  = logit_scale * N(0,1) over [B,K,V]; per (b,k) ``boost_count`` distinct ids, drawn uniformly, get
    ``+U(boost_lo, boost_hi)``;
  * h0 ~ N(0,1) [B,H], kept fp32;
  * W_ih [3H,E] ~ N(0, 1/sqrt(E)); W_hh [3H,H] ~ N(0, 1/sqrt(H)); b_ih, b_hh [3H] ~ N(0, 1/sqrt(H));
  * emb [V,E] ~ N(0, 0.02); W_c [V,H] ~ N(0, 0.1);
  * everything is drawn in fp32 and, for the bf16 workloads, cast to bf16 by round-to-nearest-even. The cast tensor
    is the input of both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import torch

# Workload table. ``dtype`` is the storage type of the logits and of every weight.
CONFIGS: Dict[int, dict] = {
    0: dict(name="tiny-oracle-check", B=1, V=1024, K=4, M=8, H=32, E=32, n=8, max_depth=4, T=0.0,
            dtype="f32", logit_scale=3.0, boost_count=16, boost_lo=4.0, boost_hi=10.0),
    1: dict(name="qwen3-4b-b1", B=1, V=151936, K=16, M=64, H=512, E=2560, n=16, max_depth=16, T=0.0,
            dtype="bf16", logit_scale=3.0, boost_count=16, boost_lo=4.0, boost_hi=10.0),
    2: dict(name="qwen3-4b-b64", B=64, V=151936, K=16, M=64, H=512, E=2560, n=16, max_depth=16, T=0.0,
            dtype="bf16", logit_scale=3.0, boost_count=16, boost_lo=4.0, boost_hi=10.0),
    3: dict(name="qwen3-8b-b32", B=32, V=151936, K=16, M=64, H=1024, E=4096, n=32, max_depth=16, T=0.5,
            dtype="bf16", logit_scale=3.0, boost_count=16, boost_lo=4.0, boost_hi=10.0),
    4: dict(name="stress-b256", B=256, V=151936, K=16, M=128, H=512, E=2560, n=64, max_depth=16, T=1.0,
            dtype="bf16", logit_scale=1.5, boost_count=64, boost_lo=2.0, boost_hi=6.0),
}

STREAM = {"logits": 1, "boost_ids": 2, "boost_vals": 3, "h0": 4, "w_ih": 5, "w_hh": 6, "b_ih": 7, "b_hh": 8,
          "emb": 9, "w_c": 10, "lmhead_hidden": 11, "lmhead_w": 12, "attn_q": 13, "attn_k": 14, "attn_v": 15,
          "attn_tree": 16}


@dataclass
class Shape:
    B: int
    V: int
    K: int
    M: int
    H: int
    E: int
    n: int
    max_depth: int
    T: float
    dtype: str = "bf16"
    logit_scale: float = 3.0
    boost_count: int = 16
    boost_lo: float = 4.0
    boost_hi: float = 10.0
    name: str = "custom"

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} V={self.V} K={self.K} M={self.M} E={self.E} H={self.H} n={self.n} "
                f"max_depth={self.max_depth} T={self.T:g} {self.dtype}")


def shape(config: int, **overrides) -> Shape:
    return replace(Shape(**CONFIGS[config]), **overrides)


@dataclass
class Inputs:
    """One round's inputs. Tensors live on the device they were drawn on."""
    shape: Shape
    logits: torch.Tensor            # [B,K,V] f32 or bf16
    h0: torch.Tensor                # [B,H] f32
    w_ih: torch.Tensor              # [3H,E] gate rows r|z|n
    w_hh: torch.Tensor              # [3H,H] gate rows r|z|n
    b_ih: Optional[torch.Tensor]    # [3H]
    b_hh: Optional[torch.Tensor]    # [3H]
    emb: torch.Tensor               # [V,E]
    w_c: torch.Tensor               # [V,H]
    seed: int = 0
    extra: dict = field(default_factory=dict)


def _gen(device, seed: int, name: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 64 + STREAM[name])
    return g


def _normal(shape_, std: float, device, seed: int, name: str) -> torch.Tensor:
    x = torch.randn(shape_, generator=_gen(device, seed, name), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def _distinct_ids(rows: int, count: int, V: int, device, seed: int) -> torch.Tensor:
    """``count`` distinct uniform ids in [0,V) per row (rejection of repeats, in draw order)."""
    if count > V:
        raise ValueError("boost_count > V")
    g = _gen("cpu", seed, "boost_ids")
    out = torch.empty(rows, count, dtype=torch.int64)
    draw = max(2 * count, 8)
    for r in range(rows):
        chosen: list = []
        seen = set()
        while len(chosen) < count:
            cand = torch.randint(0, V, (draw,), generator=g).tolist()
            for c in cand:
                if c not in seen:
                    seen.add(c)
                    chosen.append(c)
                    if len(chosen) == count:
                        break
        out[r] = torch.tensor(chosen, dtype=torch.int64)
    return out.to(device)


def _logits_f32(s: Shape, device, seed: int) -> torch.Tensor:
    B, K, V = s.B, s.K, s.V
    logits = _normal((B, K, V), s.logit_scale, device, seed, "logits")
    if s.boost_count > 0:
        ids = _distinct_ids(B * K, s.boost_count, V, device, seed)
        g = _gen(device, seed, "boost_vals")
        boost = torch.rand((B * K, s.boost_count), generator=g, device=device, dtype=torch.float32)
        boost = boost * (s.boost_hi - s.boost_lo) + s.boost_lo
        logits.view(B * K, V).scatter_add_(1, ids, boost)
    return logits


def _resolve(config_or_shape, seed, overrides):
    if isinstance(config_or_shape, Shape):
        s = replace(config_or_shape, **overrides)
        cfg_idx = 0
    else:
        cfg_idx = int(config_or_shape)
        s = shape(cfg_idx, **overrides)
    return s, (1234 + 100 * cfg_idx if seed is None else seed)


def make_logits(config_or_shape, device="cpu", seed: Optional[int] = None, **overrides) -> torch.Tensor:
    """Only the marginal logits [B,K,V] of a workload (same values as make_inputs draws)."""
    s, seed = _resolve(config_or_shape, seed, overrides)
    logits = _logits_f32(s, torch.device(device), seed)
    return logits.to(s.torch_dtype).contiguous()


def make_inputs(config_or_shape, device="cpu", seed: Optional[int] = None, biases: bool = True,
                **overrides) -> Inputs:
    """Draw one round's inputs for a workload (an index into CONFIGS, or a Shape)."""
    s, seed = _resolve(config_or_shape, seed, overrides)
    device = torch.device(device)
    B, V, H, E = s.B, s.V, s.H, s.E

    logits = _logits_f32(s, device, seed)
    h0 = _normal((B, H), 1.0, device, seed, "h0")
    w_ih = _normal((3 * H, E), 1.0 / math.sqrt(E), device, seed, "w_ih")
    w_hh = _normal((3 * H, H), 1.0 / math.sqrt(H), device, seed, "w_hh")
    b_ih = _normal((3 * H,), 1.0 / math.sqrt(H), device, seed, "b_ih") if biases else None
    b_hh = _normal((3 * H,), 1.0 / math.sqrt(H), device, seed, "b_hh") if biases else None
    emb = _normal((V, E), 0.02, device, seed, "emb")
    w_c = _normal((V, H), 0.1, device, seed, "w_c")

    td = s.torch_dtype
    if td != torch.float32:
        # torch's float32 -> bfloat16 conversion rounds to nearest even.
        logits = logits.to(td)
        w_ih, w_hh, emb, w_c = (t.to(td) for t in (w_ih, w_hh, emb, w_c))
        b_ih = b_ih.to(td) if b_ih is not None else None
        b_hh = b_hh.to(td) if b_hh is not None else None
    return Inputs(shape=s, logits=logits.contiguous(), h0=h0.contiguous(), w_ih=w_ih.contiguous(),
                  w_hh=w_hh.contiguous(), b_ih=b_ih, b_hh=b_hh, emb=emb.contiguous(), w_c=w_c.contiguous(),
                  seed=seed)


def bits_u16(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (host copy)."""
    import numpy as np
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def host_array(t: Optional[torch.Tensor]):
    """Host numpy view of an input tensor in its storage form: uint16 bits for bf16, float32 otherwise."""
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return bits_u16(t)
    return t.detach().to("cpu").contiguous().numpy()


def make_target_next(tokens, parents, V: int, p_agree: float, seed: int = 99):
    """Synthetic greedy next tokens of a target model for verified trees (input data for the acceptance walk).

    tokens/parents [B,n] (numpy); returns [B,n+1] int32: entry 0 stands for the root, entry 1 + i for node i. With
    probability ``p_agree`` the entry is the token of one of that node's children in the tree (drawn uniformly),
    otherwise a uniform vocabulary id (a node without children always gets a uniform id)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    B, n = tokens.shape
    out = rng.integers(0, V, size=(B, n + 1), dtype=np.int64)
    for b in range(B):
        kids = [[] for _ in range(n + 1)]
        for i in range(n):
            kids[int(parents[b, i]) + 1].append(int(tokens[b, i]))
        for j in range(n + 1):
            if kids[j] and rng.random() < p_agree:
                out[b, j] = kids[j][int(rng.integers(0, len(kids[j])))]
    return out.astype(np.int32)


def make_lmhead_inputs(R: int, D: int, V: int, device="cpu", seed: int = 4321):
    """The fused projection's inputs: the backbone hidden states of R (request, block position) rows, N(0, 1), and
    an LM head of V rows, N(0, 1/sqrt(D)) (so the logits are about N(0, 1)); both drawn in fp32 from one seeded
    CPU generator, then rounded to bf16, which is the input of both the GPU path and the oracle."""
    hidden = _normal((R, D), 1.0, "cpu", seed, "lmhead_hidden").to(torch.bfloat16)
    w_head = _normal((V, D), 1.0 / math.sqrt(D), "cpu", seed, "lmhead_w").to(torch.bfloat16)
    return hidden.to(device), w_head.to(device)


def make_attention_inputs(B: int, n: int, L: int, Hq: int, Hkv: int, d: int, device="cpu", seed: int = 2468):
    """The verify pass's attention inputs: queries of the n tree nodes [B,n,Hq,d], the key and value cache rows of
    the L prefix positions and the n tree positions [B,Hkv,L+n,d] (all N(0,1) in fp32, cast to bf16), and the
    ancestor masks [B,n,n] of random prefix-closed trees (node i's parent drawn uniformly among the root and the
    nodes before it), the structure dt_build_trees emits."""
    q = _normal((B, n, Hq, d), 1.0, "cpu", seed, "attn_q").to(torch.bfloat16)
    k = _normal((B, Hkv, L + n, d), 1.0, "cpu", seed, "attn_k").to(torch.bfloat16)
    v = _normal((B, Hkv, L + n, d), 1.0, "cpu", seed, "attn_v").to(torch.bfloat16)
    g = _gen("cpu", seed, "attn_tree")
    mask = torch.zeros((B, n, n), dtype=torch.uint8)
    for b in range(B):
        par = [-1]
        for i in range(1, n):
            par.append(int(torch.randint(-1, i, (1,), generator=g).item()))
        for i in range(n):
            j = i
            while j >= 0:
                mask[b, i, j] = 1
                j = par[j]
    return q.to(device), k.to(device), v.to(device), mask.to(device)
