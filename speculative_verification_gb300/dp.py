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
