"""Host-side arithmetic for the measurement report (no GPU work here).

* causal-adjusted FLOPs: 4 d per allowed (q, k) pair (QK^T and PV, 2 d each);
  A = N(N+1)/2 allowed pairs per head under the causal mask, N^2 otherwise.
* the pipelined ring time model ([RA-CN] "通信为什么可能被隐藏": with double
  buffering a step costs about max(T_compute, T_comm), so P steps cost
  P * max(T_compute, T_comm); "一个容量与时间的估算示例" works 8 x max(3, 2) =
  24 ms and 8 x max(3, 5) = 40 ms);
* per-shard load imbalance (max/min of allowed pairs or times).
"""
from __future__ import annotations


def allowed_pairs(N: int, causal: bool) -> int:
    return N * (N + 1) // 2 if causal else N * N


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> int:
    return 4 * B * H * d * allowed_pairs(N, causal)


def pipelined_ring_ms(steps: int, t_compute_ms: float, t_comm_ms: float) -> float:
    return steps * max(t_compute_ms, t_comm_ms)


def imbalance(values) -> float:
    values = list(values)
    lo = min(values)
    return float("inf") if lo == 0 else max(values) / lo
