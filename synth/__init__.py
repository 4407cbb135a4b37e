"""Seeded synthetic inputs for the decode step: model shapes, BF16 weights, KV pools,
page tables and decode schedules.

This module holds no arithmetic of the decode step itself (no norm, projection,
attention or sampling). It only draws random numbers and lays them out. Both the
CPU oracle (``oracle/``) and the CUDA path consume the arrays it returns, so that
the two sides always see the same bits.

Distributions (all seeds explicit):
  * linear weights and router weights ~ N(0, 0.02), drawn in fp32, rounded to BF16
    with round-to-nearest-even (``torch.Tensor.to(torch.bfloat16)``);
  * RMSNorm gains = 1.0, optionally 1 + N(0, gain_noise) for tests that must
    notice a gain being ignored;
  * KV cache contents ~ N(0, 1) in BF16;
  * token ids uniform on [0, vocab); page pools are random permutations.

Each tensor gets its own sub-seed derived from (seed, layer, name), so a tensor's
values do not depend on the order in which the others are generated.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional

import numpy as np
import torch

PAGE_SIZE = 16


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Shape of a pre-norm decoder (Llama-style reading of the Cohere megakernel
    page, section "Megakernel ne demek", and the Kog page's 2B example)."""
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    n_experts: int = 0
    top_k: int = 0
    expert_ffn_dim: int = 0
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    sliding_window: int = 0
    # 0-based layer i slides iff sliding_window > 0 and i % 2 == 1
    max_batch: int = 8
    page_size: int = PAGE_SIZE
    max_positions: int = 8192 + 512

    @property
    def is_moe(self) -> bool:
        return self.n_experts > 0

    def layer_is_sliding(self) -> List[int]:
        return [1 if (self.sliding_window > 0 and i % 2 == 1) else 0
                for i in range(self.n_layers)]

    def weight_bytes(self) -> int:
        """Bytes of every BF16 tensor in the model (embedding included)."""
        d, hd = self.d_model, self.head_dim
        per_layer = (self.n_q_heads * hd * d + 2 * self.n_kv_heads * hd * d
                     + d * self.n_q_heads * hd + 2 * d)
        if self.is_moe:
            per_layer += self.n_experts * d + self.n_experts * 3 * self.expert_ffn_dim * d
        else:
            per_layer += 3 * self.ffn_dim * d
        total = self.n_layers * per_layer + 2 * self.vocab * d + d
        return 2 * total

    def with_(self, **kw) -> "ModelConfig":
        return dataclasses.replace(self, **kw)


TINY = ModelConfig("tiny", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                   ffn_dim=768, vocab=4096, max_batch=8, max_positions=512)
DENSE_2B = ModelConfig("dense-2b", n_layers=25, d_model=2048, n_q_heads=16, n_kv_heads=4,
                       head_dim=128, ffn_dim=8192, vocab=128256, max_positions=8192 + 1024)
DENSE_2B_SWA = DENSE_2B.with_(name="dense-2b-swa", sliding_window=4096)
MOE = ModelConfig("moe-64x768", n_layers=24, d_model=2048, n_q_heads=32, n_kv_heads=4,
                  head_dim=64, ffn_dim=0, vocab=128256, n_experts=64, top_k=8,
                  expert_ffn_dim=768, max_positions=4096 + 256)
DENSE_8B = ModelConfig("dense-8b", n_layers=32, d_model=4096, n_q_heads=32, n_kv_heads=8,
                       head_dim=128, ffn_dim=14336, vocab=128256, max_positions=32768 + 256)

CONFIGS: Dict[str, ModelConfig] = {c.name: c for c in (TINY, DENSE_2B, DENSE_2B_SWA, MOE, DENSE_8B)}


def sub_seed(seed: int, *parts) -> int:
    """Stable 63-bit sub-seed from a base seed and a tensor name."""
    h = hashlib.sha256(repr((int(seed),) + tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device: str, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device: str = "cpu") -> torch.Tensor:
    """N(0, std) drawn in fp32 from a seeded generator, rounded to BF16 (RNE)."""
    g = _gen(device, seed)
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=g)
    return t.to(torch.bfloat16)


def _gain(d: int, seed: int, gain_noise: float, device: str) -> torch.Tensor:
    if gain_noise <= 0.0:
        return torch.ones(d, dtype=torch.bfloat16, device=device)
    return (1.0 + normal_bf16((d,), gain_noise, seed, device).float()).to(torch.bfloat16)


def make_weights(cfg: ModelConfig, seed: int, device: str = "cpu", std: float = 0.02,
                 gain_noise: float = 0.0) -> dict:
    """All weights of ``cfg`` as BF16 tensors on ``device``.

    Linear layers are ``[out, in]`` row-major (the nn.Linear convention).
    Experts are stacked ``[E, out, in]``.
    """
    d, hd = cfg.d_model, cfg.head_dim
    W = {
        "embed": normal_bf16((cfg.vocab, d), std, sub_seed(seed, "embed"), device),
        "final_norm": _gain(d, sub_seed(seed, "final_norm"), gain_noise, device),
        "lm_head": normal_bf16((cfg.vocab, d), std, sub_seed(seed, "lm_head"), device),
        "layers": [],
    }
    for l in range(cfg.n_layers):
        s = lambda name: sub_seed(seed, l, name)  # noqa: E731
        L = {
            "attn_norm": _gain(d, s("attn_norm"), gain_noise, device),
            "wq": normal_bf16((cfg.n_q_heads * hd, d), std, s("wq"), device),
            "wk": normal_bf16((cfg.n_kv_heads * hd, d), std, s("wk"), device),
            "wv": normal_bf16((cfg.n_kv_heads * hd, d), std, s("wv"), device),
            "wo": normal_bf16((d, cfg.n_q_heads * hd), std, s("wo"), device),
            "mlp_norm": _gain(d, s("mlp_norm"), gain_noise, device),
        }
        if cfg.is_moe:
            E, Fe = cfg.n_experts, cfg.expert_ffn_dim
            L["router"] = normal_bf16((E, d), std, s("router"), device)
            L["exp_gate"] = normal_bf16((E, Fe, d), std, s("exp_gate"), device)
            L["exp_up"] = normal_bf16((E, Fe, d), std, s("exp_up"), device)
            L["exp_down"] = normal_bf16((E, d, Fe), std, s("exp_down"), device)
        else:
            F = cfg.ffn_dim
            L["w_gate"] = normal_bf16((F, d), std, s("w_gate"), device)
            L["w_up"] = normal_bf16((F, d), std, s("w_up"), device)
            L["w_down"] = normal_bf16((d, F), std, s("w_down"), device)
        W["layers"].append(L)
    return W


def weights_to(W: dict, device: str) -> dict:
    out = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in W.items()
           if k != "layers"}
    out["layers"] = [{k: v.to(device) for k, v in L.items()} for L in W["layers"]]
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor → contiguous numpy uint16 array of its bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def kv_pool_shape(cfg: ModelConfig, num_pages: int):
    """Paged KV pool layout: [layer][page][K=0 / V=1][kv head][slot][head_dim]."""
    return (cfg.n_layers, num_pages, 2, cfg.n_kv_heads, cfg.page_size, cfg.head_dim)


def fill_normal_bf16_(t: torch.Tensor, seed: int, std: float = 1.0, chunk: int = 1 << 26):
    """Fill a BF16 tensor (any device) in place with N(0, std), chunk by chunk."""
    flat = t.view(-1)
    g = _gen(t.device.type, seed)
    tmp = torch.empty(min(chunk, flat.numel()), dtype=torch.float32, device=t.device)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        tmp[:n].normal_(0.0, std, generator=g)
        flat[i:i + n].copy_(tmp[:n])
    return t


def random_page_tables(rng: np.random.Generator, num_pages: int, pages_per_seq: List[int],
                       max_pages: int) -> np.ndarray:
    """Disjoint page runs for each sequence, drawn as one random permutation of the
    pool. Entry i of row b holds the page for positions [16 i, 16 i + 16); -1 = unused."""
    need = int(sum(pages_per_seq))
    if need > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {need}")
    perm = rng.permutation(num_pages)
    pt = np.full((len(pages_per_seq), max_pages), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(pages_per_seq):
        pt[b, :n] = perm[o:o + n]
        o += n
    return pt


def prefix_shared_page_tables(rng: np.random.Generator, num_pages: int, batch: int,
                              prefix_pages: int, private_pages: int, max_pages: int) -> np.ndarray:
    """Sequences that share one page-aligned prefix run, each followed by private pages."""
    perm = rng.permutation(num_pages)
    need = prefix_pages + batch * private_pages
    if need > num_pages:
        raise ValueError("pool too small")
    pt = np.full((batch, max_pages), -1, dtype=np.int32)
    shared = perm[:prefix_pages]
    o = prefix_pages
    for b in range(batch):
        pt[b, :prefix_pages] = shared
        pt[b, prefix_pages:prefix_pages + private_pages] = perm[o:o + private_pages]
        o += private_pages
    return pt


def random_tokens(rng: np.random.Generator, vocab: int, n) -> np.ndarray:
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def replacement_slots(event_index: int, batch: int = 8):
    """Continuous-batching replacement: at the k-th event (every 64 steps), batch slots
    (2k mod B, 2k+1 mod B) finish and are refilled with fresh 512-token contexts."""
    return ((2 * event_index) % batch, (2 * event_index + 1) % batch)
