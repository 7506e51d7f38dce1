"""Data-parallel replicas: the host logic of a run on N GPUs.

The path does not shard: N processes (one per GPU) each run the whole
training step on their own synthetic batch, with no data-path collective.
What crosses processes is timing only -- every rank's timed region is
bracketed by a barrier, the job time is the slowest rank's, and the
whole-job throughput counts the work of all N replicas over that time.
The functions take the process group module so they run under NCCL on GPUs
and under gloo on CPU alike.
"""


def max_over_ranks(seconds, dist=None, device=None):
    """The largest of the ranks' timed-region lengths (seconds); the value
    itself without a process group."""
    if dist is None:
        return float(seconds)
    import torch

    x = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return float(x.item())


def whole_job_rate(work_per_step, steps, world, seconds_max):
    """Units per second of the whole job: every replica did `steps` steps of
    `work_per_step` units, finished within the slowest rank's time."""
    if seconds_max <= 0.0:
        raise ValueError("timed region must be positive")
    return world * work_per_step * steps / seconds_max


def is_reporter(rank):
    """Only rank 0 prints the result line (and runs the reference arm)."""
    return rank == 0
