"""The library under CUDA graph capture: a prefill and several decode steps recorded once into
a graph and replayed give the same bytes as the same calls made eagerly (the calls only enqueue
work on the caller's stream; nothing synchronises the host or allocates)."""
import pytest
import torch

from linear_attention_fwd_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K(cuda_device):
    from linear_attention_fwd_gb300 import build, kda
    build.build()
    return kda


def test_prefill_and_decode_replayed_from_a_graph(K):
    inp = inputs.make_prefill(batch=1, seqlen=700, heads=3, dk=128, dv=128, dtype=torch.bfloat16,
                              device="cuda", seed=501, init_state=True)
    dec = inputs.make_decode_inputs(steps=4, rows=1, heads=3, dk=128, dv=128,
                                    dtype=torch.bfloat16, device="cuda", seed=502)
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])

    def run(out, fs, st, outs):
        K.kda_chunk_fwd(*args, inp["initial_state"], out=out, final_state=fs)
        st.copy_(fs)
        for t in range(4):
            K.kda_recurrent_step(dec["q"][t], dec["k"][t], dec["v"][t], dec["g"][t],
                                 dec["beta"][t], st, out=outs[t])

    mk = lambda: (torch.empty_like(inp["v"]), torch.empty_like(inp["initial_state"]),
                  torch.empty_like(inp["initial_state"]),
                  [torch.empty((1, 3, 128), dtype=torch.bfloat16, device="cuda") for _ in range(4)])
    eager = mk()
    run(*eager)
    torch.cuda.synchronize()

    graph_bufs = mk()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside the capture (attributes, tensor maps)
        run(*graph_bufs)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for b in (graph_bufs[0], graph_bufs[1], graph_bufs[2], *graph_bufs[3]):
        b.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(*graph_bufs)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(graph_bufs[0], eager[0]) and torch.equal(graph_bufs[1], eager[1])
    assert torch.equal(graph_bufs[2], eager[2])
    for a, b in zip(graph_bufs[3], eager[3]):
        assert torch.equal(a, b)


def test_balanced_schedule_replayed_with_changing_decay(K):
    # The balanced schedule decides on the device, from the data, where each piece starts (a
    # warm-up start, or the sequence start when a key channel does not decay).  One graph
    # replayed while the decay changes under it (a channel without decay, then the standard
    # decay, in the same buffers) must give what the eager calls give, replay after replay:
    # nothing carried from one replay to the next may decide anything.
    inp = inputs.make_prefill(batch=1, seqlen=64 * 64, heads=4, dk=128, dv=128,
                              dtype=torch.bfloat16, device="cuda", seed=503)
    g_dec = inp["g"].clone()
    g_flat = g_dec.clone()
    g_flat[..., 5] = 0
    out = torch.empty_like(inp["v"])
    fs = torch.empty((1, 4, 128, 128), dtype=torch.float32, device="cuda")

    def run():
        K.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], out=out, final_state=fs)

    eager = {}
    for name, gv in (("decaying", g_dec), ("flat", g_flat)):
        inp["g"].copy_(gv)
        run()
        torch.cuda.synchronize()
        eager[name] = (out.clone(), fs.clone())
    assert not torch.equal(eager["decaying"][1], eager["flat"][1])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for name in ("flat", "decaying", "flat", "flat", "decaying", "decaying", "flat"):
        inp["g"].copy_(g_dec if name == "decaying" else g_flat)
        out.zero_()
        fs.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager[name][0]) and torch.equal(fs, eager[name][1]), name
