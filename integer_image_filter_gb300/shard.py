"""Host-side planning for running one long sequence on several GPUs.

The motion feature shards by frame ranges with no data-path collective: rank r
owns frames [s_r, e_r) and also reads the frame before its first one (a
one-frame halo), so its first SAD is against frame s_r - 1 exactly as in the
unsharded sequence.  The only cross-rank value is the score of the first frame
of the next shard, which the last frame of each shard needs for motion2
(motion2_i = min(score_i, score_{i+1})); it is exchanged once on the host.
Independent sequences (or picture pairs) need no exchange at all.  motion_v2
(the blur of prev - cur) needs exactly the same one-frame halo, so the same
shards serve it; the moment sums are per pair and split by pairs.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Shard:
    start: int      # first frame this rank reports
    end: int        # one past the last frame this rank reports
    read_from: int  # first frame this rank reads (start - 1 except for rank 0)

    @property
    def count(self) -> int:
        return self.end - self.start

    @property
    def drop_first(self) -> bool:
        """True when the first SAD computed on [read_from, end) belongs to the
        previous shard (the halo frame's own SAD) and must be dropped."""
        return self.read_from < self.start


def shard_frames(n: int, world: int, rank: int) -> Shard:
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    end = start + base + (1 if rank < extra else 0)
    read_from = start - 1 if start > 0 and end > start else start
    return Shard(start, end, read_from)


def stitch_motion2(local_sad, shard: Shard, w: int, h: int, group=None):
    """Scores and motion2 for this rank's frames.  local_sad holds SAD_i for
    i in [shard.start, shard.end) (halo SAD already dropped).  Exchanges the
    first score of every shard over torch.distributed (host tensors, any
    backend) when a process group is initialised."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from . import motion_scores_from_sad

    sad = np.ascontiguousarray(np.asarray(local_sad, dtype=np.uint64))
    score, _ = motion_scores_from_sad(sad, w, h)
    first = float(score[0]) if sad.size else float("nan")
    nxt = None
    if dist.is_available() and dist.is_initialized():
        world = dist.get_world_size(group)
        rank = dist.get_rank(group)
        t = torch.tensor([first, float(sad.size)], dtype=torch.float64)
        out = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(out, t, group=group)
        for r in range(rank + 1, world):     # the next non-empty shard
            if out[r][1].item() > 0:
                nxt = float(out[r][0].item())
                break
    return motion_scores_from_sad(sad, w, h, next_score=nxt)
