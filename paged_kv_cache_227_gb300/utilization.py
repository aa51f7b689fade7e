"""Block utilisation of a KV pool under two placement rules, host only.

A cache kept in one contiguous piece per request has to be reserved for the
request's maximum length; 16-token blocks handed out as a request grows, found
through its block table, leave less than one block of slack per request
("Serving", section 23.4 Paged Attention, and its 96-block, eight-request
demo; "Paged Attention: Managing the KV Cache Like Virtual Memory",
inference-serving tag page).  `run` replays a request schedule against a pool
under either rule, placing blocks with this library's allocator for the paged
rule, and reports per step how many requests run and how many blocks and
tokens they hold.

Rules of the replay: first come, first served admission (the head of the
queue is admitted at the start of a step when it fits; nobody passes it); the
prompt is written on admission and every running request appends one token
per step, the admission step included, until its output is complete; it is
released at the end of that step.  `reserve` places ceil(max/16) contiguous
blocks at the lowest position that fits; `paged` needs the prompt's blocks on
admission and takes one more block whenever a request crosses a block
boundary (a request that finds no free block skips that step).
"""
from dataclasses import dataclass

from . import BLOCK_SIZE, BlockAllocator


@dataclass
class Request:
    arrival: int
    prompt: int
    output: int
    max_tokens: int


@dataclass
class Step:
    step: int
    running: int
    blocks: int
    tokens: int
    admitted: int


class _Contiguous:
    """Lowest-first-fit ranges of whole blocks."""

    def __init__(self, n):
        self.used = bytearray(n)

    def place(self, k):
        run = 0
        for b, u in enumerate(self.used):
            run = 0 if u else run + 1
            if run == k:
                s = b - k + 1
                self.used[s:b + 1] = b"\x01" * k
                return s
        return None

    def release(self, s, k):
        self.used[s:s + k] = bytes(k)


def run(policy, num_blocks, requests, steps, block_size=BLOCK_SIZE):
    """Replays `requests` (Request or (arrival, prompt, output, max) tuples)
    for `steps` steps; returns (list of Step, admission step per request or
    None)."""
    reqs = [r if isinstance(r, Request) else Request(*r) for r in requests]
    if policy not in ("reserve", "paged"):
        raise ValueError("policy is 'reserve' or 'paged'")
    by_arrival = {}
    for i, r in enumerate(reqs):
        by_arrival.setdefault(r.arrival, []).append(i)
    admitted = [None] * len(reqs)
    queue, live = [], {}                 # live: request -> [generated, held]
    space = _Contiguous(num_blocks) if policy == "reserve" else None
    alloc = BlockAllocator(num_blocks, block_size) if policy == "paged" else None
    where = {}
    out = []
    for t in range(steps):
        queue.extend(by_arrival.get(t, ()))
        while queue:
            i = queue[0]
            r = reqs[i]
            if policy == "reserve":
                k = -(-r.max_tokens // block_size)
                s = space.place(k)
                if s is None:
                    break
                where[i] = (s, k)
            else:
                if alloc.num_free() < -(-r.prompt // block_size):
                    break
                alloc.seq_add(i)
                if r.prompt:
                    alloc.extend(i, r.prompt)
            queue.pop(0)
            admitted[i] = t
            live[i] = [0, r.prompt]
        for i in sorted(live):
            if alloc is not None:
                try:
                    alloc.append_slot(i)
                except MemoryError:
                    continue
            live[i][0] += 1
            live[i][1] += 1
        if policy == "reserve":
            blocks = sum(where[i][1] for i in live)
        else:
            blocks = num_blocks - alloc.num_free()
        out.append(Step(t, len(live), blocks, sum(v[1] for v in live.values()),
                        sum(a is not None for a in admitted)))
        for i in [i for i, v in live.items() if v[0] >= reqs[i].output]:
            if policy == "reserve":
                space.release(*where.pop(i))
            else:
                alloc.seq_free(i)
            del live[i]
    return out, admitted


def demo_requests():
    """The 96-block, eight-request demo as this library reads it: a request may
    grow to 384 tokens (24 blocks, so four reservations fill the pool) and
    holds at most 170; one arrives every 10 steps."""
    prompts = [30, 45, 20, 60, 35, 50, 25, 40]
    outputs = [120, 90, 150, 60, 100, 80, 130, 70]
    return [Request(10 * k, p, o, 384) for k, (p, o) in enumerate(zip(prompts, outputs))]


def utilisation(trace, block_size=BLOCK_SIZE):
    """Tokens held over token slots held, over the steps where anything runs."""
    held = sum(s.blocks for s in trace) * block_size
    return sum(s.tokens for s in trace) / held if held else 0.0
