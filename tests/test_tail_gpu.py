"""Parity of the forward's split tail (attn_fwd_ws) with the fp64 oracle.

With a workspace, the work items left over after whole rounds of one item
per SM go to a second launch that gives each CTA an equal run of their key
blocks; an item whose blocks fall to several CTAs is computed in pieces
that the last one to finish merges with the online-softmax rescaling.  The
shapes below are chosen so that items really are cut into pieces: ragged
sequence ends, the causal diagonal, several pieces per item, a tail with
and without a main launch before it, and every head dim and dtype.
Needs a GB300 (sm_103a)."""
import numpy as np
import pytest
import torch

import attn_inputs as ai
from attn_check import compare, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import warp_specialized_gb300 as ws
    ws.load_library(build_if_missing=True)
    assert torch.cuda.is_available()


def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _max_pieces(d, esize):
    """Pieces per tile whose merge the tail kernel can stage in its Q tiles
    and K/V ring (the forward kernel's shared-memory layout)."""
    tile = d * esize * 128
    nqt = 2 if (d <= 128 and tile <= 32768) else 1
    misc = 1024 + 512 + 2 * 128 * 4 + 2 * 2 * 128 * 4
    slots = min(8, (232448 - misc - 128 * 128 - nqt * tile) // tile)
    return 1 + (nqt + slots) * tile // ((d + 2) * 128 * 4)


def tail_split(B, H, N, d, causal, esize=2):
    """The host's split, restated: (main items, tail items, key blocks per
    tail CTA, tail grid, [(bh, first query tile, query tiles)] of the tail
    items)."""
    g = _num_sms()
    nqt_cta = 2 if d <= 128 else 1
    n_qt = -(-N // 128)
    n_pairs = -(-n_qt // nqt_cta)
    bh_n = B * H
    n_items = bh_n * n_pairs
    tail = n_items % g
    main = n_items - tail
    items, units = [], 0
    for it in range(main, n_items):
        if causal:
            pair, bh = n_pairs - 1 - it // bh_n, it % bh_n
        else:
            bh, pair = it // n_pairs, it % n_pairs
        qt0 = pair * nqt_cta
        walk = min(qt0 + nqt_cta, n_qt) if causal else n_qt
        units += walk
        items.append((bh, qt0, min(nqt_cta, n_qt - qt0)))
    walk_max = max((min(qt0 + nq, n_qt) if causal else n_qt) for _, qt0, nq in items) if items else 0
    pmax = _max_pieces(d, esize)
    share = max(8, (walk_max - 1 + pmax - 2) // (pmax - 1) + 2) if pmax >= 2 else walk_max
    grid = min(g, max(1, units // share)) if units else 0
    per_cta = units / grid if grid else 0.0
    return main, tail, per_cta, grid, items


def _split_rows(items, H):
    """(heads, rows) of the tail items: the heads they touch, every row of
    their query tiles."""
    heads = sorted({(bh // H, bh % H) for bh, _, _ in items})
    rows = sorted({r for _, qt0, nq in items for r in range(qt0 * 128, (qt0 + nq) * 128)})
    return heads, rows


def _check_split(B, H, N, d, dtype, causal, seed, n_random_rows=None):
    main, tail, per_cta, grid, items = tail_split(B, H, N, d, causal, 1 if dtype == "fp8" else 2)
    assert tail > 0 and grid > 0
    inp = ai.make_inputs(B, H, N, d, dtype, seed=seed)
    o, lse = run_gpu(inp, causal, split_tail=True)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all(), "unwritten output"
    heads, rows = _split_rows(items, H)
    rows = np.array([r for r in rows if r < N], dtype=np.int64)
    if n_random_rows is not None:
        rows = np.union1d(rows[:: max(1, len(rows) // 512)], sample_rows(N, n_random_rows, seed))
    if dtype == "fp8" and causal:
        # e4m3 P on a causal row of only a few keys can miss the 6e-2 bound
        # by itself, split or not (P's rounding is not in the fp64 oracle):
        # compare the rows that see at least one whole key block
        rows = rows[rows >= 127]
    compare(inp, causal, o, lse, heads=heads, rows=rows)
    # the same call without the split: the two differ only by the order in
    # which the row sums and O are accumulated
    o1, lse1 = run_gpu(inp, causal, split_tail=False)
    tol_o = 6e-2 if dtype == "fp8" else 8e-3
    assert float((o - o1).abs().max()) <= tol_o
    assert float((lse - lse1).abs().max()) <= 1e-3
    return main, per_cta


# (B, H, N, d, dtype); per case the comment gives items, tail, grid, blocks
# per tail CTA for the non-causal split
SPLIT_SMALL = [
    (1, 1, 2048, 128, "bf16"),   # 8 items, no main launch, 16 CTAs of 8 blocks
    (1, 2, 1500, 128, "bf16"),   # ragged: 12 items of 12 blocks, pieces 8 + 4
    (1, 3, 1500, 64, "bf16"),    # d = 64
    (1, 2, 1500, 128, "fp16"),
    (1, 2, 1500, 128, "fp8"),
    (1, 1, 8192, 128, "bf16"),   # 32 items of 64 blocks over 152 CTAs: ~5 pieces each
    (2, 20, 2048, 128, "bf16"),  # 320 items: a main launch of 2 rounds, then 16 split items
    (1, 1, 300, 128, "bf16"),    # 2 tiles, one item: under 8 blocks, one CTA
]


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", SPLIT_SMALL, ids=lambda x: str(x))
def test_split_items_small(B, H, N, d, dtype, causal):
    _check_split(B, H, N, d, dtype, causal, seed=500 + N + d + H)


def test_d256_runs_whole_items():
    """d = 256 keeps Q in Tensor Memory and its shared-memory tile in the
    K/V ring, which leaves no room for a piece merge: it takes no workspace,
    is never advised a split, and a requested split runs whole items."""
    import warp_specialized_gb300 as ws
    assert ws.attn_fwd_workspace_size(256, ws.ATTN_BF16) == 0
    assert ws.attn_fwd_workspace_size(256, ws.ATTN_FP8_E4M3) == 0
    assert not ws.attn_fwd_split_advised(1, 1, 8192, 256, False, ws.ATTN_BF16)
    for causal in (False, True):
        inp = ai.make_inputs(1, 2, 1500, 256, "bf16", seed=1756 + causal)
        o, lse = run_gpu(inp, causal, split_tail=True)
        compare(inp, causal, o, lse)


def test_split_cuts_items():
    """The small cases above do cut items: some tail CTA's range of key
    blocks starts inside an item (ranges restated from the host's plan:
    CTA c starts at c * U / G, plus the ramp behind a main launch)."""
    cut = 0
    for B, H, N, d, dtype in SPLIT_SMALL:
        for causal in (False, True):
            main, tail, per_cta, grid, items = tail_split(B, H, N, d, causal,
                                                          1 if dtype == "fp8" else 2)
            n_qt = -(-N // 128)
            walks = [(min(qt0 + (2 if d <= 128 else 1), n_qt) if causal else n_qt)
                     for _, qt0, _ in items]
            starts, acc = set(), 0
            for w_ in walks:
                starts.add(acc)
                acc += w_
            units = acc
            ramp = min(units // grid // 4, 4) if main > 0 else 0
            f = [(c * units * grid + ramp * c * (grid - c)) // (grid * grid) for c in range(grid)]
            if any(x not in starts for x in f):
                cut += 1
    assert cut >= 10, cut


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_split_items_full_size(dtype, causal):
    """B2 H16 N8192 d128: 1024 items, 6 whole rounds, 112 split ones."""
    main, _ = _check_split(2, 16, 8192, 128, dtype, causal, seed=77, n_random_rows=64)
    assert main > 0


def test_split_is_deterministic():
    """The pieces are merged in a fixed order, so repeated calls give the
    same bits whichever CTA finishes last."""
    inp = ai.make_inputs(1, 1, 8192, 128, "bf16", seed=9)
    o0, l0 = run_gpu(inp, False, split_tail=True)
    for _ in range(3):
        o1, l1 = run_gpu(inp, False, split_tail=True)
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_workspace_checks():
    import warp_specialized_gb300 as ws
    dev = torch.device("cuda", 0)
    q = torch.randn(1, 1, 1024, 128, device=dev, dtype=torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 1024, device=dev)
    need = ws.attn_fwd_workspace_size(128, ws.ATTN_BF16)
    assert need > 0
    assert ws.attn_fwd_workspace_size(128, ws.ATTN_FP32) == 0
    assert ws.attn_fwd_workspace_size(96, ws.ATTN_BF16) == 0
    buf = torch.empty(need + 512, dtype=torch.uint8, device=dev)
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 1024,
            128, 0.088, False, ws.ATTN_BF16)
    s = torch.cuda.current_stream().cuda_stream
    assert ws.attn_fwd_ws_raw(*args, buf.data_ptr(), need - 1, s) == 1   # short
    assert ws.attn_fwd_ws_raw(*args, 0, need, s) == 1                    # null
    assert ws.attn_fwd_ws_raw(*args, buf.data_ptr() + 16, need, s) == 3  # misaligned
    assert ws.attn_fwd_ws_raw(*args, buf.data_ptr(), need, s) == 0
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0


def test_caller_workspace_reused():
    """One caller workspace serves calls of different shapes in a row."""
    import warp_specialized_gb300 as ws
    dev = torch.device("cuda", 0)
    buf = torch.empty(ws.attn_fwd_workspace_size(128, ws.ATTN_BF16), dtype=torch.uint8,
                      device=dev)
    for (B, H, N), causal in [((1, 1, 2048), False), ((1, 2, 1500), True), ((1, 1, 2048), True)]:
        inp = ai.make_inputs(B, H, N, 128, "bf16", seed=N + causal)
        o, lse = run_gpu(inp, causal, split_tail=True, workspace=buf)
        compare(inp, causal, o, lse)


def test_split_advice():
    """The split is advised where the problem is one partial round (fewer
    items than SMs) whose longest item is well above a tail CTA's share plus
    the split's own cost; not behind whole rounds, nor where there is no
    leftover."""
    import warp_specialized_gb300 as ws
    g = _num_sms()
    bf = ws.ATTN_BF16
    assert g == 152, "the shapes below assume 152 SMs"
    assert ws.attn_fwd_split_advised(1, 1, 8192, 128, False, bf)      # 32 items of 64 blocks
    assert ws.attn_fwd_split_advised(1, 2, 8192, 128, True, bf)       # 64 items, one round
    assert ws.attn_fwd_split_advised(1, 4, 8192, 128, True, bf)       # causal, 128 items
    assert not ws.attn_fwd_split_advised(1, 16, 8192, 128, False, bf)  # 3 rounds + 56 items
    assert not ws.attn_fwd_split_advised(2, 16, 8192, 128, False, bf)  # 112 of 1024: even
    assert not ws.attn_fwd_split_advised(1, 16, 8192, 128, True, bf)   # causal behind rounds
    assert not ws.attn_fwd_split_advised(1, 4, 8192, 128, False, bf)   # 128 items: share 54
    assert not ws.attn_fwd_split_advised(1, 2, 1500, 128, False, bf)   # short items
    assert not ws.attn_fwd_split_advised(g, 1, 256, 128, False, bf)    # whole rounds only
    assert not ws.attn_fwd_split_advised(2, 16, 8192, 96, False, bf)   # invalid d
    assert not ws.attn_fwd_split_advised(2, 16, 8192, 128, False, ws.ATTN_FP32)
