"""Batch sharding across GPUs.

Slot-heads are independent (no exchange step in the recurrence), so several
GPUs decode disjoint shards of the batch with no collective on the data path.
Requests are kept whole: a request and every branch forked from it land on the
same rank, because a branch indexes its request's dense base in that GPU's
memory.
"""


def shard_requests(num_requests, world, rank):
    """Contiguous block of request ids owned by `rank` (sizes differ by <= 1)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(num_requests, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def slots_of_requests(requests, branches_per_request):
    """Local slot layout of a shard: requests first, then their branches,
    request-major.  Returns (request_slots, branch_slots[list per request])."""
    reqs = list(requests)
    r_slots = list(range(len(reqs)))
    b0 = len(reqs)
    b_slots = [[b0 + i * branches_per_request + j for j in range(branches_per_request)]
               for i in range(len(reqs))]
    return r_slots, b_slots
