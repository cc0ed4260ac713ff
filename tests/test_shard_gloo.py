"""The N>1 host path on CPU: frame-range shards with a one-frame halo and the
motion2 stitch across ranks, as world_size-2 gloo processes.  The SADs a rank
would compute on its GPU are stood in for by the oracle's (the shard logic is
what is under test)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from integer_image_filter_gb300.shard import shard_frames


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("n,world", [(10, 2), (11, 3), (2, 2), (1, 2), (0, 3), (7, 1)])
def test_shards_cover_each_frame_once(n, world):
    got = []
    for r in range(world):
        s = shard_frames(n, world, r)
        assert s.read_from in (s.start, s.start - 1)
        got += list(range(s.start, s.end))
    assert got == list(range(n))


def _worker(rank, world, port, frames, want_score, want_m2, result_q, variant="motion"):
    import torch.distributed as dist

    import oracle
    from integer_image_filter_gb300 import _build, load_library
    from integer_image_filter_gb300.shard import shard_frames, stitch_motion2
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        _build.build()
        load_library()
        o = oracle.Oracle()
        n, h, w = frames.shape
        sh = shard_frames(n, world, rank)
        seq = o.motion_v2_sequence if variant == "motion_v2" else o.motion_sad_sequence
        sad = seq(np.ascontiguousarray(frames[sh.read_from:sh.end]), 8)
        if sh.drop_first:
            sad = sad[1:]
        score, m2 = stitch_motion2(sad, sh, w, h)
        ok = (np.array_equal(score, want_score[sh.start:sh.end])
              and np.array_equal(m2, want_m2[sh.start:sh.end]))
        result_q.put((rank, ok))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("variant", ["motion", "motion_v2"])
def test_sharded_sequence_matches_unsharded(variant):
    import oracle
    import synth
    frames = synth.smooth_sequence(21, 9, 64, 40, 2)
    o = oracle.Oracle()
    sad = (o.motion_v2_sequence if variant == "motion_v2" else o.motion_sad_sequence)(frames, 8)
    want_score, want_m2 = o.scores(sad, 64, 40)
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, frames, want_score, want_m2, q,
                                               variant))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    results = dict(q.get(timeout=10) for _ in range(world))
    assert all(p.exitcode == 0 for p in procs)
    assert results == {0: True, 1: True}
