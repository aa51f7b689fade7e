"""Reference block-utilisation simulation in plain Python.

TEST INFRASTRUCTURE (see the package docstring).

A server cannot know how long an answer will be, so a cache kept in one
contiguous piece is reserved for the worst case; 16-token blocks handed out as
a sequence grows, through a block table, waste less than one block per
sequence ("Serving", section 23.4 Paged Attention; "Paged Attention: Managing
the KV Cache Like Virtual Memory", inference-serving tag page).  The section's
demo: a pool of 96 blocks serves eight requests that arrive over time and grow
token by token; reserving each maximum lets only four run, paging runs every
request when it arrives.

Readings (the pages give no request parameters and no admission rule):
  * A request (arrival step, prompt tokens, output tokens, maximum tokens)
    is admitted first come, first served: the head of the waiting queue is
    admitted at the start of a step if the policy can place it, and nothing
    behind it jumps ahead.
  * On admission its prompt is written at once; each later step, including
    the admission step, appends one generated token until its output is
    complete; it is then freed at the end of that step.
  * reserve: admission needs ceil(max_tokens / 16) contiguous free blocks
    (lowest first fit) and holds them to the end.
  * paged: admission needs the prompt's blocks; later blocks are taken one at
    a time from the reference allocator's FIFO free list as the request grows.
    A request that cannot get its next block waits in place (the step does
    not append for it); the demo never runs out.
The trace per step: admitted requests, running requests, blocks held, tokens
held.
"""
from oracle.allocator import ReferenceAllocator

BS = 16


def blocks_for(tokens, bs=BS):
    return -(-tokens // bs)


def simulate(policy, num_blocks, requests, steps, bs=BS):
    """requests: list of (arrival, prompt, output, max_tokens).  Returns a
    list of per-step dicts and the admission step of each request."""
    n = len(requests)
    admitted = [None] * n
    waiting = []
    running = {}          # request -> tokens generated so far
    held = {}             # request -> tokens held
    free_map = [True] * num_blocks   # reserve policy
    ranges = {}
    alloc = ReferenceAllocator(num_blocks, bs) if policy == "paged" else None
    trace = []
    for t in range(steps):
        waiting += [r for r in range(n) if requests[r][0] == t]
        # admissions, first come first served
        while waiting:
            r = waiting[0]
            _, prompt, _, mx = requests[r]
            if policy == "reserve":
                need = blocks_for(mx, bs)
                start = None
                run = 0
                for b in range(num_blocks):
                    run = run + 1 if free_map[b] else 0
                    if run == need:
                        start = b - need + 1
                        break
                if start is None:
                    break
                for b in range(start, start + need):
                    free_map[b] = False
                ranges[r] = (start, need)
            else:
                if alloc.num_free() < blocks_for(prompt, bs):
                    break
                alloc.seq_add(r)
                for _ in range(prompt):
                    alloc.append_slot(r)
            waiting.pop(0)
            admitted[r] = t
            running[r] = 0
            held[r] = prompt
        # one generated token per running request
        for r in sorted(running):
            if policy == "paged":
                try:
                    alloc.append_slot(r)
                except MemoryError:
                    continue
            running[r] += 1
            held[r] += 1
        blocks = (sum(ranges[r][1] for r in running) if policy == "reserve"
                  else num_blocks - alloc.num_free())
        trace.append({"step": t, "running": len(running), "blocks": blocks,
                      "tokens": sum(held[r] for r in running),
                      "admitted": sum(1 for a in admitted if a is not None)})
        for r in [r for r in running if running[r] >= requests[r][2]]:
            if policy == "reserve":
                s0, k = ranges.pop(r)
                for b in range(s0, s0 + k):
                    free_map[b] = True
            else:
                alloc.seq_free(r)
            del running[r], held[r]
    return trace, admitted


def demo_requests():
    """The 96-block, 8-request demo with this build's reading of its sizes:
    a request may grow to 384 tokens (24 blocks, so 4 reservations fill the
    pool) but holds at most 170; one arrives every 10 steps."""
    prompts = [30, 45, 20, 60, 35, 50, 25, 40]
    outputs = [120, 90, 150, 60, 100, 80, 130, 70]
    return [(10 * k, p, o, 384) for k, (p, o) in enumerate(zip(prompts, outputs))]
