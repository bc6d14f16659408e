"""CUDA-graph capture and the in-kernel shrink -> expand dependency across launches.

One launch runs the shrink units and the fused units; a fused unit's expand waits for its
tile's ready flag. The flags are cleared by the last CTA of each launch, so a launch never
sees a flag left by an earlier one: consecutive calls and replays of a captured graph each
wait for their own shrink. A test-only option holds every flag back for a while, so an
expand that did not wait would read the previous call's U rows and give wrong output."""
import pytest
import torch

from mixed_lora_projection_gb300.synth import WORKLOADS, Workload, make_inputs

from gpu_util import TOL, oracle_rows, rel_err, run, sample_rows

pytestmark = pytest.mark.gpu

DELAY_US = 300


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    return torch.device("cuda", 0)


def _ll(w):
    from mixed_lora_projection_gb300 import LoraLinear
    return LoraLinear(w.d_in, w.d_out, w.rank, w.T, 16, 0)


def _fresh_x(inp, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    inp.x.copy_(torch.randn(inp.x.shape, generator=g).to(torch.bfloat16))


@pytest.mark.parametrize("cluster", [1, 2])
def test_delayed_flags_are_awaited_across_calls(dev, cluster):
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["sweep_qkv_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, cluster)
        want = []
        for seed in (1, 2):
            _fresh_x(inp, seed)
            want.append(run(ll, inp, off, ids).clone())
        ll.set_option(L.OPT_DEBUG_PUBLISH_DELAY_US, DELAY_US)
        for seed, ref in zip((1, 2), want):
            _fresh_x(inp, seed)
            y = run(ll, inp, off, ids)
            torch.cuda.synchronize()
            assert ll.status() == 0
            assert torch.equal(y, ref)


def test_graph_replays_match_eager_calls(dev):
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["sweep_qkv_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    seeds = (11, 12, 13)
    with _ll(w) as ll:
        want = []
        for seed in seeds:
            _fresh_x(inp, seed)
            want.append(run(ll, inp, off, ids).clone())
        y = torch.empty_like(want[0])
        ll.set_option(L.OPT_DEBUG_PUBLISH_DELAY_US, DELAY_US)
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            run(ll, inp, off, ids, y=y)          # same shape once before capture
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(ll, inp, off, ids, y=y)
        for rep in range(2):
            for seed, ref in zip(seeds, want):
                _fresh_x(inp, seed)              # device buffers are read at every replay
                y.zero_()
                g.replay()
                torch.cuda.synchronize()
                assert torch.equal(y, ref), (rep, seed)
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=64, seed=3)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], oracle_rows(inp, off, ids, rows)) <= TOL


def test_capture_of_a_call_with_an_uploaded_work_list_is_refused(dev):
    from mixed_lora_projection_gb300 import LoraError, _lib as L
    w = WORKLOADS["prefill_16k"]          # 128 row tiles: the work list is uploaded per call
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = run(ll, inp, off, ids).clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            marker = torch.zeros(1, device=dev)
            marker += 1
            with pytest.raises(LoraError) as e:
                run(ll, inp, off, ids, y=y)
        assert e.value.code == L.LORA_EUNSUPPORTED
        torch.cuda.synchronize()
        y2 = run(ll, inp, off, ids)            # the handle still works eagerly
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y, y2)


def test_four_bit_base_graph_replays(dev):
    # the 4-bit-base path (shrink launch + 4-bit kernel) recorded once and replayed with fresh X
    from mixed_lora_projection_gb300 import w4_repack
    from mixed_lora_projection_gb300.synth import Workload, make_w4_base
    import numpy as np
    lens, ids = [48, 200, 8], [0, 1, 0]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4g", 31, off[-1], 512, 1024, 64, tuple(off), tuple(ids), scales=(0.75,))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = w4_repack(q)
    with _ll(w) as ll:
        want = []
        for seed in (41, 42):
            _fresh_x(inp, seed)
            want.append(ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone())
        y = torch.empty_like(want[0])
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales, y=y)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales, y=y)
        for seed, ref in zip((41, 42, 41), (want[0], want[1], want[0])):
            _fresh_x(inp, seed)
            y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(y, ref)
        assert ll.status() == 0


def test_one_launch_calls_beside_a_busy_stream(dev):
    # one-launch calls (fused units wait for other CTAs' shrink units) issued while another
    # stream keeps the GPU busy with long matmuls: the launch starts only when its whole grid
    # can be resident, so with a 20 ms wait limit every call still completes and matches
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["sweep_qkv_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    a = torch.randn(8192, 8192, device=dev).to(torch.bfloat16)
    with _ll(w) as ll:
        ref = run(ll, inp, off, ids).clone()
        torch.cuda.synchronize()
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        busy = torch.cuda.Stream(dev)
        busy.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(busy):
            c = a
            for _ in range(60):
                c = (c @ a) * 1e-2                     # tens of ms of full-GPU work
        ys = [run(ll, inp, off, ids).clone() for _ in range(6)]
        torch.cuda.synchronize()
        assert ll.status() == 0
    for y in ys:
        assert torch.equal(y, ref)


def test_two_handles_on_two_streams(dev):
    # two handles' one-launch calls interleaved on two streams (each grid waits only on itself)
    from mixed_lora_projection_gb300 import _lib as L
    w1, w2 = WORKLOADS["sweep_qkv_multi"], WORKLOADS["sweep_o_multi"]
    in1, in2 = make_inputs(w1, dev), make_inputs(w2, dev)
    o1, i1, o2, i2 = list(w1.seg_offsets), list(w1.seg_ids), list(w2.seg_offsets), list(w2.seg_ids)
    with _ll(w1) as l1, _ll(w2) as l2:
        r1, r2 = run(l1, in1, o1, i1).clone(), run(l2, in2, o2, i2).clone()
        torch.cuda.synchronize()
        for ll in (l1, l2):
            ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s1.wait_stream(torch.cuda.current_stream(dev))
        s2.wait_stream(torch.cuda.current_stream(dev))
        y1, y2 = [], []
        for _ in range(8):
            with torch.cuda.stream(s1):
                y1.append(run(l1, in1, o1, i1).clone())
            with torch.cuda.stream(s2):
                y2.append(run(l2, in2, o2, i2).clone())
        torch.cuda.synchronize()
        assert l1.status() == 0 and l2.status() == 0
    assert all(torch.equal(y, r1) for y in y1) and all(torch.equal(y, r2) for y in y2)


def test_programmatic_dependent_launch_keeps_every_dependency(dev):
    # a chain in which every call reads the previous call's Y as its X, through two handles
    # (5,120 -> 6,144 and back; the second splits K in halves for these 48-row batches): with
    # LORA_OPT_PDL each kernel starts on the SMs the previous one leaves, requests its first W
    # tiles and waits for it before anything else, so every output equals the chain run without
    # it, eagerly and replayed from a CUDA graph
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    T = 48
    wa = Workload("pdl_a", 21, T, 5120, 6144, 16, (0, T), (0,))
    wb = Workload("pdl_b", 22, T, 6144, 5120, 16, (0, T), (0,))
    ia, ib = make_inputs(wa, dev), make_inputs(wb, dev)
    x0 = ia.x.clone()
    with LoraLinear(5120, 6144, 16, T, 8, 0) as ha, LoraLinear(6144, 5120, 16, T, 8, 0) as hb:
        def chain(pdl, outs):
            for h in (ha, hb):
                h.set_option(L.OPT_PDL, pdl)
            x = x0
            for i in range(6):
                h, inp = (ha, ia) if i % 2 == 0 else (hb, ib)
                x = h.forward(x, [0, T], [0], inp.w, inp.a, inp.b, inp.scales, y=outs[i])
            return outs
        shapes = [(T, 6144) if i % 2 == 0 else (T, 5120) for i in range(6)]
        ref = chain(0, [torch.empty(s, dtype=torch.bfloat16, device=dev) for s in shapes])
        ref = [y.clone() for y in ref]
        eager = chain(1, [torch.empty(s, dtype=torch.bfloat16, device=dev) for s in shapes])
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ref, eager))
        bufs = [torch.zeros(s, dtype=torch.bfloat16, device=dev) for s in shapes]
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            chain(1, bufs)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        for b in bufs:
            b.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain(1, bufs)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ref, bufs))
        assert ha.status() == 0 and hb.status() == 0
