"""Stream semantics of the C ABI: calls are stream-ordered and asynchronous on the context's stream.

- Two contexts on two streams, with all their work in flight at once, give the same histograms as
  one context run alone.
- acf_set_stream moves a context to another stream between calls.
- A warmed-up acf_correlate (its workspace already allocated) can be captured into a CUDA graph
  and replayed. The replays give the captured call's results.
- The library's own graph replay of repeated calls (option "graphs"): the same results and launch
  counts as calls launched one by one, the inputs' current contents read, acf_get_info describing
  the replayed call, kernel timing recording every replayed launch, and calls launched one by one
  again when an option changes or the option is off.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture(scope="module")
def data(acf):
    a = synth.catalogs(6000, 5000, 10, 30.0, seed=81)
    b = synth.catalogs(4000, 4500, 6, 60.0, seed=82)
    ref = {}
    ctx = acf.Context(0)
    for name, c in (("a", a), ("b", b)):
        t = tuple(map(_dev, (c.ra_d, c.dec_d, c.ra_r, c.dec_r)))
        out = ctx.correlate(*t, 0.25, 720)
        torch.cuda.synchronize()
        ref[name] = (t, [acf.as_uint64(h).copy() for h in out[:3]], out[3].cpu().numpy())
    ctx.close()
    return ref


def test_two_contexts_on_two_streams_at_once(acf, data):
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    c1, c2 = acf.Context(0, s1), acf.Context(0, s2)
    try:
        outs = []
        for _ in range(3):  # several rounds, nothing synchronised in between
            with torch.cuda.stream(s1):
                o1 = c1.correlate(*data["a"][0], 0.25, 720)
            with torch.cuda.stream(s2):
                o2 = c2.correlate(*data["b"][0], 0.25, 720)
            outs.append((o1, o2))
        torch.cuda.synchronize()
        for o1, o2 in outs:
            for o, name in ((o1, "a"), (o2, "b")):
                for h, r in zip(o[:3], data[name][1]):
                    assert np.array_equal(acf.as_uint64(h), r)
                assert np.allclose(o[3].cpu().numpy(), data[name][2], rtol=0, atol=0, equal_nan=True)
    finally:
        c1.close()
        c2.close()


def test_set_stream_moves_a_context(acf, data):
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ctx = acf.Context(0, s1)
    try:
        with torch.cuda.stream(s1):
            o1 = ctx.correlate(*data["a"][0], 0.25, 720)
        s2.wait_stream(s1)
        acf.acf_set_stream(ctx.handle, s2)
        ctx.stream = s2
        with torch.cuda.stream(s2):
            o2 = ctx.correlate(*data["b"][0], 0.25, 720)
        torch.cuda.synchronize()
        for o, name in ((o1, "a"), (o2, "b")):
            for h, r in zip(o[:3], data[name][1]):
                assert np.array_equal(acf.as_uint64(h), r)
    finally:
        ctx.close()


def test_correlate_captured_in_a_cuda_graph(acf, data):
    s = torch.cuda.Stream()
    ctx = acf.Context(0, s)
    try:
        t, ref, ref_om = data["a"]
        outs = tuple(torch.empty(720, dtype=torch.int64, device="cuda") for _ in range(3)) + (
            torch.empty(720, dtype=torch.float64, device="cuda"),)
        with torch.cuda.stream(s):
            ctx.correlate(*t, 0.25, 720, out=outs)  # warm-up: allocates the workspace
        s.synchronize()
        for o in outs:
            o.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ctx.correlate(*t, 0.25, 720, out=outs)
        for _ in range(3):
            for o in outs:
                o.zero_()
            g.replay()
            torch.cuda.synchronize()
            for h, r in zip(outs[:3], ref):
                assert np.array_equal(acf.as_uint64(h), r)
            assert np.allclose(outs[3].cpu().numpy(), ref_om, rtol=0, atol=0, equal_nan=True)
    finally:
        ctx.close()


def test_repeated_calls_replay_a_graph(acf, data):
    s = torch.cuda.Stream()
    ctx = acf.Context(0, s)
    try:
        t, ref, ref_om = data["a"]
        with torch.cuda.stream(s):
            outs = tuple(torch.empty(720, dtype=torch.int64, device="cuda") for _ in range(3)) + (
                torch.empty(720, dtype=torch.float64, device="cuda"),)

        def call():
            with torch.cuda.stream(s):
                for o in outs:
                    o.zero_()
                k0 = ctx.info("kernel_launches")
                ctx.correlate(*t, 0.25, 720, out=outs)
            s.synchronize()
            return ctx.info("kernel_launches") - k0

        def check(r=ref, om=ref_om):
            for h, x in zip(outs[:3], r):
                assert np.array_equal(acf.as_uint64(h), x)
            assert np.allclose(outs[3].cpu().numpy(), om, rtol=0, atol=0, equal_nan=True)

        base = ctx.info("graph_replays")
        launches = []
        for _ in range(4):  # the first call runs as usual, the second is captured, then replays
            launches.append(call())
            check()
        assert ctx.info("graph_replays") - base == 3
        assert len(set(launches)) == 1, launches
        assert ctx.info("layout") == 1 and ctx.info("launches") == 1 and ctx.info("exact_flagged") > 0

        # the graph reads the inputs' current contents: other catalogs of the same sizes
        c2 = synth.catalogs(6000, 5000, 4, 90.0, seed=83)
        t2 = tuple(map(_dev, (c2.ra_d, c2.dec_d, c2.ra_r, c2.dec_r)))
        ref_ctx = acf.Context(0)
        o2 = ref_ctx.correlate(*t2, 0.25, 720)
        torch.cuda.synchronize()
        ref2 = [acf.as_uint64(h).copy() for h in o2[:3]]
        om2 = o2[3].cpu().numpy()
        ref_ctx.close()
        with torch.cuda.stream(s):
            for dst, src in zip(t, t2):
                dst.copy_(src)
        n0 = ctx.info("graph_replays")
        call()
        assert ctx.info("graph_replays") == n0 + 1
        check(ref2, om2)
        # the fixture's inputs back in place (other tests share them)
        a = synth.catalogs(6000, 5000, 10, 30.0, seed=81)
        with torch.cuda.stream(s):
            for dst, src in zip(t, (a.ra_d, a.dec_d, a.ra_r, a.dec_r)):
                dst.copy_(torch.from_numpy(np.ascontiguousarray(src)).cuda())

        # another option: launched one by one, then captured when it repeats; the first graph stays
        ctx.set_option("exact", 0)
        n0 = ctx.info("graph_replays")
        call()
        call()
        assert ctx.info("graph_replays") == n0 + 1 and ctx.info("exact_flagged") == 0
        ctx.set_option("exact", 2)
        call()
        assert ctx.info("graph_replays") == n0 + 2
        check()

        # kernel timing: a graph of its own (its timing events are nodes of it), and every pair
        # kernel of every call timed, replays included
        ctx.set_option("kernel_timing", 1)
        n0 = ctx.info("graph_replays")
        for _ in range(4):
            assert call() == launches[0]
            check()
        assert ctx.info("graph_replays") == n0 + 3
        kt = ctx.kernel_times()
        assert len(kt) == 12 and all(x > 0 for x in kt), kt  # DD, DR, RR of four calls
        # the same with the fix-ups timed (a graph of its own again)
        ctx.set_option("kernel_timing", 2)
        n0 = ctx.info("graph_replays")
        for _ in range(4):
            call()
            check()
        assert ctx.info("graph_replays") == n0 + 3
        kt = ctx.kernel_times()
        assert len(kt) == 12 and all(x > 0 for x in kt), kt
        ctx.set_option("kernel_timing", 0)
        # the option off: every kernel launched by itself
        ctx.set_option("graphs", 0)
        n0 = ctx.info("graph_replays")
        assert call() == launches[0]
        check()
        assert ctx.info("graph_replays") == n0
        ctx.set_option("graphs", 1)
    finally:
        ctx.close()


def test_repeated_host_calls_replay_a_graph_with_page_locked_buffers(acf, data):
    # acf_correlate_host with page-locked host buffers: the copies join the kernels in the graph;
    # with pageable ones (which a graph cannot hold) every call runs launch by launch
    s = torch.cuda.Stream()
    ctx = acf.Context(0, s)
    try:
        c = synth.catalogs(6000, 5000, 10, 30.0, seed=81)  # the fixture's catalogs "a"
        ref, ref_om = data["a"][1], data["a"][2]
        host_in = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in (c.ra_d, c.dec_d, c.ra_r, c.dec_r)]
        host_out = [torch.empty(720, dtype=torch.int64).pin_memory() for _ in range(3)] + [
            torch.empty(720, dtype=torch.float64).pin_memory()]
        base = ctx.info("graph_replays")
        for _ in range(4):
            for o in host_out:
                o.zero_()
            acf.acf_correlate_host(ctx.handle, host_in[0], host_in[1], c.n_d, host_in[2], host_in[3], c.n_r, 0.25, 720,
                                   *host_out)
            for h, r in zip(host_out[:3], ref):
                assert np.array_equal(acf.as_uint64(h), r)
            assert np.allclose(host_out[3].numpy(), ref_om, rtol=0, atol=0, equal_nan=True)
        assert ctx.info("graph_replays") - base == 3
        out = (np.empty(720, np.uint64), np.empty(720, np.uint64), np.empty(720, np.uint64), np.empty(720, np.float64))
        n0 = ctx.info("graph_replays")
        for _ in range(3):
            dd, dr, rr, om = ctx.correlate_host(c.ra_d, c.dec_d, c.ra_r, c.dec_r, 0.25, 720, out=out)
            for h, r in zip((dd, dr, rr), ref):
                assert np.array_equal(h, r)
        assert ctx.info("graph_replays") == n0
    finally:
        ctx.close()
