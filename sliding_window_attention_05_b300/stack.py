"""The hybrid attention stack: layers that alternate SWA(w, s) with full causal
attention, each with its own KV cache, run as prefill followed by per-token
decode steps.

The layer pattern follows "Hybrid Sliding Window Attention (Hybrid SWA)",
section "一、2. Hybrid SWA 的设计机制" (sliding-window layers interleaved with
global-attention layers), and the SWAA explainer of arXiv 2608.28444, section
"核心方法" (alternate layers keep full attention; SWA layers use w = 2048 with
s = 100 sinks). A full-causal layer is SWA with a window that covers every
position the run will reach (w = prompt length + decode steps) and no sinks, so
its ring cache never evicts: the same kernels serve both kinds of layer.

A layer can also run in the SWAA "FA decode" mode (the SWAA page, "如何将Sliding
Window Attention Adaptation应用到你的LLM项目中", its list of methods, item 1, and
the `force_fa_decode` switch of section "配置SWAA：参数详解"): the prompt is
prefilled with SWA(w, s), but every position is kept and each decoded token
attends to the whole history with full causal attention. Its cache is then a
ring whose window covers every position the run reaches (w_cache = max_len,
no sinks), so it never evicts, and decode over it is full attention.

Only attention is modelled: there are no projections or weights, so each layer
receives its own q/k/v. Every computation runs in libswa.so (prefill, cache
append, fused append + decode); this module only sequences the calls.
"""
from __future__ import annotations

import torch

from . import RingCache, swa_prefill


def hybrid_layer_windows(n_layers: int, prompt_len: int, decode_steps: int, w: int = 2048,
                         s: int = 100) -> list[tuple[int, int]]:
    """(w, s) per layer: even layers SWA(w, s), odd layers full causal, written
    as SWA(prompt_len + decode_steps, 0)."""
    full = (prompt_len + decode_steps, 0)
    return [(w, s) if i % 2 == 0 else full for i in range(n_layers)]


class AttentionLayer:
    """One attention layer: SWA(w, s) prefill of a prompt, then one fused
    append + decode per new token over the layer's ring cache.

    fa_decode=True: the prompt is still prefilled with SWA(w, s), but decode
    uses full causal attention over every earlier position; max_len (prompt
    plus decode steps) sizes the non-evicting cache, which then holds
    max_len * Hkv * d bf16 per sequence for K and for V."""

    def __init__(self, B: int, Hq: int, Hkv: int, d: int, w: int, s: int,
                 scale: float | None = None, device=None, fa_decode: bool = False,
                 max_len: int | None = None):
        self.B, self.Hq, self.Hkv, self.d, self.w, self.s = B, Hq, Hkv, d, w, s
        self.scale = scale
        self.fa_decode = bool(fa_decode)
        if self.fa_decode:
            if max_len is None or max_len < 1:
                raise ValueError("fa_decode needs max_len >= 1 (prompt + decode steps)")
            # a window over every position the run reaches and no sinks: the
            # ring never evicts, so the decode key set is every earlier position
            self.cache_w, self.cache_s = int(max_len), 0
        else:
            self.cache_w, self.cache_s = w, s
        self.cache = RingCache(B, Hkv, d, self.cache_w, self.cache_s, device)

    def prefill(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out=None,
                stream=None) -> torch.Tensor:
        """Attention of every prompt position with SWA(w, s); the prompt's keys
        and values then go into the cache (only the ones that survive eviction
        are written; with fa_decode, all of them)."""
        if self.fa_decode and self.cache.length + q.shape[1] > self.cache_w:
            raise ValueError(f"prompt of {q.shape[1]} tokens exceeds max_len {self.cache_w}")
        o = swa_prefill(q, k, v, self.w, self.s, self.scale, out=out, stream=stream)
        self.cache.append(k, v, stream)
        return o

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, out=None,
             stream=None) -> torch.Tensor:
        """q [B, Hq, d], k_new/v_new [B, Hkv, d]: append the token, attend at its
        position (over K(pos) of SWA(w, s), or over every position with fa_decode)."""
        if self.fa_decode and self.cache.length >= self.cache_w:
            raise ValueError(f"decode past max_len {self.cache_w}")
        return self.cache.step(q, k_new, v_new, self.scale, out, stream)


class HybridStack:
    """A stack of AttentionLayer objects with the hybrid window pattern.

    fa_decode=True switches the sliding-window layers to the SWAA FA-decode
    mode (SWA(w, s) prefill, full-attention decode); max_len then sizes their
    caches."""

    def __init__(self, B: int, Hq: int, Hkv: int, d: int, windows: list[tuple[int, int]],
                 scale: float | None = None, device=None, fa_decode: bool = False,
                 max_len: int | None = None):
        if fa_decode and max_len is None:
            raise ValueError("fa_decode needs max_len (prompt + decode steps)")
        self.layers = [AttentionLayer(B, Hq, Hkv, d, w, s, scale, device,
                                      fa_decode=fa_decode and (max_len is None or w < max_len),
                                      max_len=max_len)
                       for w, s in windows]

    def prefill(self, qkv: list[tuple[torch.Tensor, torch.Tensor, torch.Tensor]],
                stream=None) -> list[torch.Tensor]:
        """qkv[i] = (q, k, v) of layer i, [B, L, H, d]; returns each layer's output."""
        if len(qkv) != len(self.layers):
            raise ValueError(f"expected {len(self.layers)} layers of inputs, got {len(qkv)}")
        return [layer.prefill(q, k, v, stream=stream) for layer, (q, k, v) in zip(self.layers, qkv)]

    def step(self, tokens: list[tuple[torch.Tensor, torch.Tensor, torch.Tensor]], outs=None,
             stream=None) -> list[torch.Tensor]:
        """One decode step through every layer: tokens[i] = (q, k_new, v_new) of
        layer i for the new position. outs (optional) are reused output buffers."""
        if len(tokens) != len(self.layers):
            raise ValueError(f"expected {len(self.layers)} layers of tokens, got {len(tokens)}")
        outs = outs or [None] * len(self.layers)
        return [layer.step(q, kn, vn, out=o, stream=stream)
                for layer, (q, kn, vn), o in zip(self.layers, tokens, outs)]
