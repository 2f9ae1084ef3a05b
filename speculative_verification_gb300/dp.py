"""Host-side logic of data-parallel (row-sharded) runs.

Rows are independent: the processed logits, the kept set and the draw of a
row depend only on that row's logits and parameters, and the Philox counter
is keyed by the row's own seed, position and request index.  So a batch can
be split across GPUs by rows with no collective on the data path; each rank
samples its own rows.  The only cross-rank traffic is the benchmark's
barrier and its max-over-ranks reduction of the elapsed time.
"""


def shard_rows(num_rows, rank, world):
    """Contiguous row range [start, stop) of `rank` among `world` ranks; the
    first num_rows % world ranks take one extra row."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank %d outside a world of %d" % (rank, world))
    base, extra = divmod(int(num_rows), int(world))
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def ring_seed(config, rank, index):
    """Seed of input set `index` of `rank`'s benchmark ring: distinct over
    ranks and indices (weak scaling: every rank samples its own batches)."""
    return int(config) + 7919 * (int(rank) * 1000 + int(index))


def aggregate_rate(units_per_step, steps, world, max_elapsed_ms):
    """Whole-job throughput: the units all ranks processed divided by the
    slowest rank's elapsed time."""
    if max_elapsed_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return float(units_per_step) * int(steps) * int(world) / (max_elapsed_ms / 1e3)


def free_port():
    """A TCP port on 127.0.0.1 that was free a moment ago."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def rank_env(rank, world, port, base=None):
    """The environment of one rank: what torch.distributed.run sets for a
    single-node job (RANK, LOCAL_RANK, WORLD_SIZE, LOCAL_WORLD_SIZE,
    MASTER_ADDR = 127.0.0.1, MASTER_PORT)."""
    import os
    env = dict(os.environ if base is None else base)
    env.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), LOCAL_WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    return env


def launch_local(world, argv, port=None, timeout=None):
    """Runs `argv` as `world` processes on this node, one rank each (rank r on
    local device r), and waits for all of them.  Returns 0 when every rank
    exited 0, else the first non-zero exit code; when one rank fails the
    others are stopped (they would wait for it at the next collective)."""
    import subprocess
    import time
    if world < 1:
        raise ValueError("world size must be positive")
    port = port or free_port()
    procs = [subprocess.Popen(list(argv), env=rank_env(r, world, port)) for r in range(world)]
    t0 = time.time()
    code = 0
    try:
        while procs:
            for p in list(procs):
                rc = p.poll()
                if rc is None:
                    continue
                procs.remove(p)
                if rc != 0 and code == 0:
                    code = rc
                    for q in procs:
                        q.terminate()
            if timeout is not None and time.time() - t0 > timeout:
                for q in procs:
                    q.terminate()
                return code or 124
            time.sleep(0.05)
    finally:
        for q in procs:
            if q.poll() is None:
                q.kill()
    return code
