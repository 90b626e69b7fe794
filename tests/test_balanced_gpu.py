"""GPU parity of the balanced schedule (the library's choice for dense batches on the
tensor-core kernel) against the oracle.

The schedule flattens the units' chunks in sequence-major order into W items and gives each
of G = min(SMs, W) CTAs a contiguous share, drawn on the host so that the largest cost (items,
plus an assumed 4-chunk warm-up when a share starts inside a sequence, plus half a chunk per
further piece) is as small as bisection finds; a CTA runs one piece per (sequence, head) its
share touches, a piece that starts inside a sequence warms up as a segment does (zero state past
the 2^-160 transition bound, else from the sequence start), and the piece holding a unit's last
chunk writes its final state.  Checked here: pieces that start and end inside sequences (several
per CTA) with the standard decay and an initial state, short sequences (whole sequences per
CTA), a decay-free channel (no horizon: every piece runs from the sequence start and the result
equals one CTA per unit bit for bit), a channel that stops decaying for part of each sequence
(some pieces warm up, the others run from the start), agreement with one CTA per unit at full
size, and the bounded-wait expiry path (every output and final state NaN, the status reported).
"""
import numpy as np
import pytest
import torch

from linear_attention_fwd_gb300 import inputs
from tests.parity import check_prefill, compare_prefill, f64

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def run(K, inp, **kw):
    out, sT = K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              inp.get("initial_state"), inp.get("cu_seqlens"), impl="tc", **kw)
    torch.cuda.synchronize()
    return out, sT


def rel_diff(a, b):
    a, b = f64(a), f64(b)
    return float(np.abs(a - b).max() / np.sqrt(np.mean(b * b)))


def schedule(W, nc, G):
    """Host restatement of the library's schedule: the CTAs' share boundaries x_0 .. x_G."""
    warm, piece, min_tail = 4.0, 0.5, 8

    def fill(T):
        x, xs = 0, []
        for _ in range(G):
            xs.append(x)
            cost, start = (warm if x % nc else 0.0), x
            while x < W:
                r = nc - x % nc
                extra = piece if x != start else 0.0
                if cost + extra + r <= T:
                    x, cost = x + r, cost + extra + r
                    continue
                take = int(T - cost - extra)
                if take > 0 and (x == start or take >= min_tail):
                    x += take
                break
        return x, xs + [W]
    lo, hi = W / G, W / G + nc + warm + piece + 1.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        lo, hi = (lo, mid) if fill(mid)[0] >= W else (mid, hi)
    return fill(hi)[1]


def pieces_split_inside_units(K, inp):
    """How many CTA shares start inside a unit."""
    B, T, H, _ = inp["q"].shape
    nc = (T + 63) // 64
    W = B * H * nc
    G = K.kda_chunk_fwd_auto_ctas(K.chunk_dims(inp["q"], inp["v"]), False, sms())
    assert G == min(W, sms())
    xs = schedule(W, nc, G)
    assert xs[0] == 0 and xs[-1] == W and all(a <= b for a, b in zip(xs, xs[1:]))
    return sum(1 for b in range(1, G) if xs[b] < xs[b + 1] and xs[b] % nc != 0)


def test_pieces_inside_sequences_with_the_standard_decay(K):
    # 2 x 5 units of 40 chunks (the last one partial): 400 items over the SMs, so most shares
    # start and end inside a sequence
    inp = inputs.make_prefill(batch=2, seqlen=2530, heads=5, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=401, init_state=True)
    assert pieces_split_inside_units(K, inp) > 50
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_short_sequences_snap_to_sequence_boundaries(K):
    # 3-chunk sequences: whole sequences per CTA, no splits
    inp = inputs.make_prefill(batch=40, seqlen=150, heads=6, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=402, init_state=True)
    assert pieces_split_inside_units(K, inp) == 0
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_no_horizon_runs_every_piece_from_the_sequence_start(K):
    # one channel never decays: pieces that start inside a sequence recompute it from its start
    # with the initial state, which is exactly what one CTA per unit computes
    inp = inputs.make_prefill(batch=1, seqlen=2600, heads=6, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=403, g_mode="near_bound", init_state=True)
    inp["g"][..., 7] = 0
    assert pieces_split_inside_units(K, inp) > 0
    out1, sT1 = run(K, inp, segments=1)
    out, sT = run(K, inp)
    assert torch.equal(out, out1) and torch.equal(sT, sT1)
    check_prefill(compare_prefill(inp, out1, sT1), BF)


def test_decay_free_stretch_inside_each_sequence(K):
    # 4 units of 128 chunks over the SMs (shares of ~3-4 chunks); channel 7 does not decay in
    # chunks 40-89 of every sequence.  Pieces whose 16-chunk look-back lies in that stretch have
    # no warm-up start and run from the sequence start; the rest warm up.
    inp = inputs.make_prefill(batch=2, seqlen=128 * 64, heads=2, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=405, init_state=True)
    inp["g"][:, 40 * 64:90 * 64, :, 7] = 0
    assert pieces_split_inside_units(K, inp) > 100
    out, sT = run(K, inp)
    assert torch.isfinite(out.float()).all() and torch.isfinite(sT).all()
    check_prefill(compare_prefill(inp, out, sT), BF)


def test_full_size_agrees_with_one_cta_per_unit(K):
    # B=4 H=32 T=8192: 16384 items over the SMs; heads 0 and 31 of every sequence against the
    # oracle, all heads against one CTA per unit
    inp = inputs.make_workload("prefill_b4_h32_t8192", device="cuda")
    out, sT = run(K, inp)
    out1, sT1 = run(K, inp, segments=1)
    assert rel_diff(sT, sT1) <= 1e-3
    assert rel_diff(out, out1) <= 2e-2
    check_prefill(compare_prefill(inp, out, sT, heads=[0, 31]), BF)


def test_expired_waits_under_the_balanced_schedule(K):
    inp = inputs.make_prefill(batch=2, seqlen=2530, heads=5, dk=128, dv=128, dtype=BF,
                              device="cuda", seed=404, init_state=True)
    out, sT = run(K, inp, wait_polls=0)
    assert torch.isnan(sT).all() and torch.isnan(out.float()).all()
    assert K.kda_device_status() == K.KDA_ERR_TIMEOUT
    out, sT = run(K, inp)
    assert K.kda_device_status() == K.KDA_OK
    check_prefill(compare_prefill(inp, out, sT), BF)


# ---------------------------------------------------------------- packed sequences
def packed_splits(K, lengths, H):
    """Host restatement of the device-side packed shares: how many start inside a unit."""
    items = [max((L + 63) // 64, 1) for L in lengths]
    units = [(n, h) for n in range(len(lengths)) for h in range(H)]
    starts, acc = [], 0
    for n, _ in units:
        starts.append(acc)
        acc += items[n]
    W = acc
    G = K.kda_chunk_fwd_auto_ctas(K.KdaDims(batch=1, seqlen=sum(lengths), num_seqs=len(lengths), heads=H,
                                            dk=128, dv=128, dtype=1), True, sms())

    def snap(x):
        if x >= W:
            return W
        u = max(i for i, s0 in enumerate(starts) if s0 <= x)
        c, it = x - starts[u], items[units[u][0]]
        return starts[u] if c <= 4 else (starts[u] + it if it - c <= 4 else x)
    xs = [snap(b * W // G) for b in range(G + 1)]
    assert all(a <= b for a, b in zip(xs, xs[1:])) and xs[-1] == W
    return sum(1 for b in range(1, G) if xs[b] < xs[b + 1] and xs[b] not in starts)


def test_packed_pieces_inside_sequences(K):
    # long, short, one-token and empty members: shares start inside the long ones
    lengths = [3000, 1, 0, 130, 2000, 65, 64, 700]
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=3, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=405, init_state=True, lengths=lengths)
    assert packed_splits(K, lengths, 3) > 20
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT), BF)
    torch.testing.assert_close(sT[2], inp["initial_state"][2], rtol=0, atol=0)   # the empty one
    out1, sT1 = run(K, inp, segments=1)
    assert rel_diff(sT, sT1) <= 1e-3


def test_packed_no_horizon_equals_one_cta_per_unit(K):
    lengths = [2600, 5, 1400, 0, 900]
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=4, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=406, g_mode="near_bound", init_state=True, lengths=lengths)
    inp["g"][..., 11] = 0
    assert packed_splits(K, lengths, 4) > 0
    out1, sT1 = run(K, inp, segments=1)
    out, sT = run(K, inp)
    assert torch.equal(out, out1) and torch.equal(sT, sT1)


def test_packed_more_sequences_than_threads(K):
    # 600 sequences: the device's scans over them run in more than one pass of 512
    rng = np.random.default_rng(407)
    lengths = [int(x) for x in rng.integers(0, 150, size=600)]
    inp = inputs.make_prefill(batch=1, seqlen=0, heads=2, dk=128, dv=128, dtype=BF, device="cuda",
                              seed=408, init_state=True, lengths=lengths)
    out, sT = run(K, inp)
    check_prefill(compare_prefill(inp, out, sT, heads=[1]), BF)
    out1, sT1 = run(K, inp, segments=1)
    assert rel_diff(sT, sT1) <= 1e-3
