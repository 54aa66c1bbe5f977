"""Host-side arithmetic for the measurement report (no GPU work here).

* causal-adjusted FLOPs: 4 d per allowed (q, k) pair (QK^T and PV, 2 d each);
  A = N(N+1)/2 allowed pairs per head under the causal mask, N^2 otherwise.
* the pipelined ring time model ([RA-CN] "通信为什么可能被隐藏": with double
  buffering a step costs about max(T_compute, T_comm), so P steps cost
  P * max(T_compute, T_comm); "一个容量与时间的估算示例" works 8 x max(3, 2) =
  24 ms and 8 x max(3, 5) = 40 ms);
* per-shard load imbalance (max/min of allowed pairs or times), the
  per-shard allowed-pair closed forms of the three layouts, and the time of
  a synchronous ring whose every step waits for its slowest shard ([GRA] "The
  causal mask wrecks the load balance"; [RA-CN] "Causal Attention
  让环不再完全对称").
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


def shard_positions(layout: str, n: int, P: int, r: int) -> list:
    """Global token positions of the n local rows of shard r: contiguous
    r n + i; striped i P + r (token t on shard t mod P); zigzag the chunks r
    and 2P - 1 - r of n/2 tokens, in that order."""
    if layout == "striped":
        return [i * P + r for i in range(n)]
    if layout == "zigzag":
        c = n // 2
        return [r * c + i for i in range(c)] + [(2 * P - 1 - r) * c + i for i in range(c)]
    return [r * n + i for i in range(n)]


def shard_pairs_closed_form(layout: str, n: int, P: int) -> list:
    """Causal allowed (query, key) pairs of each shard over the whole ring.
    Contiguous: shard r meets r full blocks and its diagonal, r n^2 + n(n+1)/2.
    Striped: r + 1 blocks with k <= i and P - 1 - r with k < i,
    (r + 1) n(n+1)/2 + (P - 1 - r) n(n-1)/2.  Zigzag (chunks of c = n/2):
    every off-diagonal block holds 2c^2 pairs and the diagonal 2c^2 + c, so
    2Pc^2 + c on every shard."""
    if layout == "contiguous":
        return [r * n * n + n * (n + 1) // 2 for r in range(P)]
    if layout == "striped":
        return [(r + 1) * n * (n + 1) // 2 + (P - 1 - r) * n * (n - 1) // 2 for r in range(P)]
    c = n // 2
    return [2 * P * c * c + c] * P


def synchronous_ring_ms(step_shard_ms) -> float:
    """A ring step ends when its slowest shard is done (every shard then
    passes its block on), so the ring takes sum over steps of the maximum over
    shards; step_shard_ms[s][r] is shard r's time at step s."""
    return sum(max(row) for row in step_shard_ms)
