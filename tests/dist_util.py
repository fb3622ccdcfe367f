"""Runs a function on `world` local processes joined by a torch.distributed
gloo group (127.0.0.1, a free port), with a time limit: used by the CPU tests
of the multi-process host logic and by the GPU tests that run several ranks
as processes on one GPU (the ranks exchange only host tensors; no kernel
waits on another)."""

from __future__ import annotations

import os
import socket
import traceback

import torch.multiprocessing as mp


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _entry(fn, rank, world, port, args, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        try:
            q.put((rank, "ok", fn(rank, world, *args)))
        finally:
            dist.destroy_process_group()
    except BaseException as e:  # reported to the parent, which decides
        q.put((rank, "raised", (type(e).__name__, str(e), traceback.format_exc())))


def run_ranks(fn, world: int, args=(), timeout: float = 180.0) -> dict:
    """{rank: ("ok", value) | ("raised", (type, message, traceback))}.
    fn(rank, world, *args) must be a module-level function.  A process still
    running after `timeout` seconds is killed and the call fails."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_entry, args=(fn, r, world, port, args, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(world):
            rank, kind, val = q.get(timeout=timeout)
            out[rank] = (kind, val)
    finally:
        for p in procs:
            p.join(10)
            if p.is_alive():
                p.kill()
                p.join(5)
    assert len(out) == world, f"only ranks {sorted(out)} reported within {timeout} s"
    return out
