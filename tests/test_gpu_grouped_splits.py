"""GPU parity: decode batches whose sequences read the same blocks.

With groups of 8 query heads, sequences that read the same 32 blocks in a
complete 512-token split are computed together: each K/V tile of that split is
read once per KV head for up to 8 sequences ("大模型部署.md" §2.1, PageAttention:
parallel-sampling branches share the prompt's blocks through reference counts).
These tests build block tables with such sharing directly (families of
sequences that share a prefix of blocks, nested forks, runs longer than 8,
plain sequences between them) and compare every output with the float64
oracle over the same tables.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import attention  # noqa: E402
from tests.gpu_parity import TOL, out_f64  # noqa: E402

pytestmark = pytest.mark.gpu

BS = 16


@pytest.fixture(scope="module")
def dev(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib.device_error(clear=True)
    return torch.device("cuda")


def build(seed, hq, hkv, d, seqs, scale=0.5):
    """seqs: list of (family, shared_blocks, ctx).  Sequences of one family
    read the family's prompt blocks for their first `shared_blocks` blocks and
    private blocks after that (family None: all blocks private).  Returns the
    tables, context lengths, q and the two caches (bf16 bit patterns)."""
    rng = np.random.default_rng(seed)
    need_prompt = {}
    for fam, sh, ctx in seqs:
        if fam is not None:
            need_prompt[fam] = max(need_prompt.get(fam, 0), sh)
    n_private = sum(-(-ctx // BS) - (sh if fam is not None else 0) for fam, sh, ctx in seqs)
    nb = sum(need_prompt.values()) + n_private + 8
    ids = iter(rng.permutation(nb).tolist())
    prompt = {fam: [next(ids) for _ in range(n)] for fam, n in sorted(need_prompt.items())}
    width = max(-(-ctx // BS) for _, _, ctx in seqs)
    tables = np.full((len(seqs), width), -1, dtype=np.int32)
    for s, (fam, sh, ctx) in enumerate(seqs):
        nblk = -(-ctx // BS)
        row = (prompt[fam][:sh] if fam is not None else []) + []
        while len(row) < nblk:
            row.append(next(ids))
        tables[s, :nblk] = row[:nblk]
    ctx = np.array([c for _, _, c in seqs], dtype=np.int32)
    k = workloads._values(rng, (nb, hkv, BS, d), "bf16", scale)
    v = workloads._values(rng, (nb, hkv, BS, d), "bf16", scale)
    q = workloads._values(rng, (len(seqs), hq, d), "bf16", scale)
    return tables, ctx, q, k, v


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run(lib, tables, ctx, q, k, v, hq):
    kd, vd, qd = to_dev(k), to_dev(v), to_dev(q)
    out = torch.empty_like(qd)
    lib.paged_attention_decode(out, qd, kd, vd, lib.cache_desc(kd, hq),
                               torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(),
                               int(ctx.max()))
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out


def check(lib, tables, ctx, q, k, v, hq):
    out = run(lib, tables, ctx, q, k, v, hq)
    ref = attention.decode(q, k, v, tables, ctx, BS, "bf16")
    err = np.abs(out_f64(out) - ref)
    mx, mean = TOL["bf16"]
    assert err.max() <= mx and err.mean() <= mean, (err.max(), err.mean())
    return out


# (family, shared blocks, context length) per sequence, in batch order
CASES = {
    # two branches sharing 70 blocks: splits 0 and 1 shared, split 2 partly
    "pair": [(0, 70, 70 * BS + 37), (0, 70, 70 * BS + 200)],
    # a run of 9 over 5 shared splits (a group of 8 and a single), a plain
    # sequence before and after, and a family of 3 sharing one split
    "run_of_nine": ([(None, 0, 3000)] + [(1, 170, 170 * BS + 1 + i * 7) for i in range(9)]
                    + [(None, 0, 700)] + [(2, 40, 40 * BS + 5 + i) for i in range(3)]),
    # nested forks: the third branch shares only the first split, so the runs
    # differ from split to split
    "nested": [(3, 100, 100 * BS + 9), (3, 100, 100 * BS + 100), (3, 40, 40 * BS + 60),
               (3, 100, 100 * BS + 3), (3, 100, 100 * BS + 300)],
    # context lengths on split boundaries, a long plain sequence in the middle
    "boundaries": [(4, 64, 1024), (4, 64, 1024), (4, 64, 1025), (None, 0, 20000),
                   (5, 32, 512 + 1), (5, 32, 1023), (5, 32, 1024)],
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_shared_splits_match_oracle(dev, lib, name):
    tables, ctx, q, k, v = build(11, 64, 8, 128, CASES[name])
    check(lib, tables, ctx, q, k, v, 64)


def test_shared_splits_head_dim_64(dev, lib):
    tables, ctx, q, k, v = build(12, 16, 2, 64, CASES["run_of_nine"] + CASES["nested"])
    check(lib, tables, ctx, q, k, v, 16)


def test_identical_rows_give_identical_bits(dev, lib):
    """Rows with the same table, length and q give the same bits, whether their
    only split is a grouped one (context exactly 512) or one of several."""
    seqs = [(0, 32, 512)] * 3 + [(1, 96, 96 * BS)] * 2 + [(None, 0, 900)]
    tables, ctx, q, k, v = build(13, 64, 8, 128, seqs)
    q[1] = q[0]
    q[2] = q[0]
    q[4] = q[3]
    out = check(lib, tables, ctx, q, k, v, 64)
    assert torch.equal(out[0], out[1]) and torch.equal(out[0], out[2])
    assert torch.equal(out[3], out[4])


def test_grouping_does_not_change_other_sequences(dev, lib):
    """A plain sequence's bits do not depend on shared splits elsewhere in the batch."""
    base = [(None, 0, 2500), (None, 0, 777)]
    tables, ctx, q, k, v = build(14, 64, 8, 128, base + CASES["run_of_nine"])
    alone = run(lib, tables[:2], ctx[:2], q[:2], k, v, 64)
    both = run(lib, tables, ctx, q, k, v, 64)
    assert torch.equal(alone, both[:2])
