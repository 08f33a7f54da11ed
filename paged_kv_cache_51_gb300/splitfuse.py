"""Multi-step mixed batches: a request stream turned into SplitFuse steps.

Each step spends one token budget (C++ composer, pkv_splitfuse_compose): every
running request that has finished its prompt decodes one token, then waiting
prompts take chunks in arrival order; a long prompt continues over several
steps.  The scheduler emits, per step, the pool operations that place the
step's tokens ("add" for a request's first chunk, "grow" otherwise), the batch
layout [(request, qlen)] in query-row order, and the value rows of the step's
queries.  runner.DeviceCache executes the operations.
"""

from . import pkv_splitfuse_compose


class Scheduler:
    def __init__(self, trace, token_budget):
        self.t = trace
        self.budget = token_budget
        n = len(trace.prompt_len)
        self.prompt_done = [0] * n
        self.generated = [0] * n
        self.step_no = 0

    def finished(self):
        t = self.t
        return all(self.prompt_done[i] == t.prompt_len[i] and self.generated[i] == t.gen_len[i]
                   for i in range(len(t.prompt_len)))

    def next_step(self):
        """Returns (ops, batch, q_row_indices) for this step, or None when all is done."""
        t = self.t
        n = len(t.prompt_len)
        decoding = [i for i in range(n) if self.prompt_done[i] == t.prompt_len[i]
                    and self.generated[i] < t.gen_len[i]]
        waiting = [i for i in range(n) if t.arrival[i] <= self.step_no
                   and self.prompt_done[i] < t.prompt_len[i]]
        n_dec, chunks, _ = pkv_splitfuse_compose(
            self.budget, len(decoding), [t.prompt_len[i] - self.prompt_done[i] for i in waiting])
        ops, batch, qrows = [], [], []
        for i in decoding[:n_dec]:
            pos = t.prompt_len[i] + self.generated[i]
            ops.append(("grow", i, 1, t.row_offset[i] + pos))
            batch.append((i, 1))
            qrows.append(t.row_offset[i] + pos)
            self.generated[i] += 1
        for i, c in zip(waiting, chunks):
            if c == 0:
                continue
            pos = self.prompt_done[i]
            ops.append(("add", i, c, t.row_offset[i]) if pos == 0 else
                       ("grow", i, c, t.row_offset[i] + pos))
            batch.append((i, c))
            qrows += range(t.row_offset[i] + pos, t.row_offset[i] + pos + c)
            self.prompt_done[i] += c
        self.step_no += 1
        if not batch:
            return None if self.finished() else ([], [], [])
        return ops, batch, qrows
