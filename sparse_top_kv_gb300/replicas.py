"""Several GPUs: replicas with a request partition.

The decode path shards by request: each request's index row, hot region,
dgi/lru state and host-pool rows are independent of every other request's
(vLLM HiSparse walkthrough, hisparse_swap_in_kernel: one CTA per request,
no cross-request state), so N GPUs run N independent copies of the step with
no exchange on the data path.  What crosses ranks is host-side bookkeeping
only: which requests a rank serves, the max-over-ranks time of a timed
region, and (for reporting) the summed hit/miss counters.

Everything here works on any torch.distributed backend (nccl on GPUs, gloo
on the host), and does nothing when no process group is initialised.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist


def _world() -> tuple[int, int]:
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(), dist.get_rank()
    return 1, 0


def partition_requests(num_reqs: int, world: int, rank: int) -> range:
    """Strong scaling: the contiguous, balanced share of `num_reqs` requests
    that `rank` of `world` serves (the first num_reqs % world ranks take one
    more).  The shares are disjoint and cover every request."""
    if world <= 0 or not 0 <= rank < world or num_reqs < 0:
        raise ValueError("bad partition arguments")
    base, extra = divmod(num_reqs, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def rank_request_order(num_reqs: int, rank: int) -> np.ndarray:
    """Weak scaling: every rank serves its own batch of `num_reqs` requests.
    Rank 0 keeps the generator's order; rank r > 0 takes a seeded permutation
    of it, so that ranks do not read the same host rows in the same order."""
    if rank == 0:
        return np.arange(num_reqs)
    return np.random.default_rng(1000 + rank).permutation(num_reqs)


def max_over_ranks(x: float) -> float:
    """The largest `x` over all ranks (the job's time is its slowest rank's)."""
    world, _ = _world()
    if world == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(counters: torch.Tensor) -> torch.Tensor:
    """Element-wise sum of an integer counter tensor (e.g. the hit/miss
    statistics) over ranks, for reporting; returns a new tensor on the
    counter's device."""
    world, _ = _world()
    out = counters.clone()
    if world > 1:
        dist.all_reduce(out, op=dist.ReduceOp.SUM)
    return out


def whole_job_throughput(units_per_rank: int, world: int, max_ms: float) -> float:
    """Units per second of the whole job: every rank processed
    `units_per_rank` units, and the job took the slowest rank's `max_ms`."""
    if max_ms <= 0:
        raise ValueError("max_ms must be positive")
    return world * units_per_rank / (max_ms / 1e3)
