"""Algorithmic work of the MoE layer: the numerators of its roofline.

Counts only what the layer must do, never padding or re-reads:
  * an expert is 3 FP8 matrices (gate, up: inter x hidden; down: hidden x inter)
    plus one fp32 multiplier per 128x128 block;
  * a prefill layer does 2 * 3 * hidden * inter FLOP per (token, expert) pair,
    with top_k routed pairs and n_shared shared pairs per token;
  * a decode layer must read every touched expert's weights once.
Shapes follow the KTransformers deep dive (section 1.2) and the CPU-GPU hybrid
inference article (Stream-Loading Prefill section: 3 FP8 linear modules of
7168 x 2048 per expert).
"""
from __future__ import annotations

import numpy as np


def expert_params(hidden: int, inter: int) -> int:
    return 3 * hidden * inter


def expert_bytes(hidden: int, inter: int) -> int:
    """FP8 codes plus fp32 block multipliers of one expert."""
    return expert_params(hidden, inter) + 3 * (hidden // 128) * (inter // 128) * 4


def layer_expert_bytes(hidden: int, inter: int, n_experts: int, n_shared: int = 0, shared_inter: int = 0) -> int:
    return n_experts * expert_bytes(hidden, inter) + n_shared * expert_bytes(hidden, shared_inter or inter)


def layer_flops(T: int, hidden: int, inter: int, top_k: int, n_shared: int = 1, shared_inter: int = 0) -> int:
    """Expert GEMM FLOP of one layer over T tokens (router excluded)."""
    si = shared_inter or inter
    return 2 * 3 * hidden * (inter * T * top_k + si * T * n_shared)


def router_flops(T: int, hidden: int, n_experts: int) -> int:
    return 2 * T * hidden * n_experts


def tokens_per_routed_expert(batch: int, top_k: int, n_experts: int) -> float:
    return batch * top_k / n_experts


def expected_distinct_experts(T: int, top_k: int, n_experts: int) -> float:
    """E[#experts chosen by at least one of T tokens] under uniform routing."""
    return n_experts * (1.0 - (1.0 - top_k / n_experts) ** T)


def touched_experts(ids: np.ndarray, n_experts: int) -> int:
    return int(np.unique(np.asarray(ids).reshape(-1)).size)


def decode_weight_bytes(ids: np.ndarray, hidden: int, inter: int, n_experts: int,
                        n_shared: int = 1, shared_inter: int = 0) -> int:
    """Bytes a decode step must stream: every touched routed expert plus the
    shared expert(s), counted from the realised routing."""
    return touched_experts(ids, n_experts) * expert_bytes(hidden, inter) + \
        n_shared * expert_bytes(hidden, shared_inter or inter)


def decode_gate_up_bytes(ids: np.ndarray, hidden: int, inter: int, n_experts: int,
                         n_shared: int = 1, shared_inter: int = 0) -> int:
    """The gate+up share of decode_weight_bytes (2 of the 3 matrices)."""
    per = lambda i: 2 * hidden * i + 2 * (hidden // 128) * (i // 128) * 4
    return touched_experts(ids, n_experts) * per(inter) + n_shared * per(shared_inter or inter)
