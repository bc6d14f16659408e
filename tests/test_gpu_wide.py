"""Wide row tiles (LORA_OPT_TILE_N of 272 to 512 on SM pairs; the launch-shape model takes 288 to
320 where they fill a projection's waves, LORA_OPT_WIDE_TILES): each 16-wide K step of a unit
takes a second MMA over the output columns past 256, into one accumulator of up to 512 columns.
Checked against the fp64 oracle and bit for bit against 256-column row tiles of the same handle
(the sums keep their order whatever the tile width), over second MMAs of 16 to 256 columns,
ragged column tails, K past the last 64-wide step, one and two adapters, base tiles paired with
adapter tiles, the model's own choice at full size, graph replays, programmatic dependent launch,
a wait that runs out, and the options that rule them out."""
import numpy as np
import pytest
import torch

from mixed_lora_projection_gb300.synth import WORKLOADS, Workload, make_inputs

from gpu_util import TOL, oracle_full, oracle_rows, rel_err, run, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    return torch.device("cuda", 0)


def _ll(w, max_segments=16):
    from mixed_lora_projection_gb300 import LoraLinear
    return LoraLinear(w.d_in, w.d_out, w.rank, w.T, max_segments, 0)


def _tile_n(ll, T, off, ids):
    return ll.describe(T, off, ids)["tile_n"]


# (T, d_in, d_out, r, lengths, ids, tile_n): second MMAs of 16 (272), 32 (288), 64 (320), 144
# (400) and 256 columns (512); column tails (1000 = 3 x 288 + 136: the tail's columns sit in
# both MMAs' ranges); K of 200 (three 64-wide steps and a part); a base tile paired with an
# adapter tile; two adapters; rank 256 (shrink units of 256 columns beside the wide units)
CASES = [
    (600, 320, 1000, 32, [100, 300, 200], [0, 1, 2], 288),
    (300, 256, 544, 64, [300], [1], 272),
    (520, 384, 1024, 256, [8] * 6 + [472], [0] * 6 + [1], 512),
    (257, 200, 712, 24, [257], [0], 400),
    (1024, 512, 2000, 128, [300, 400, 324], [1, 0, 2], 320),
    (129, 320, 600, 16, [60, 69], [0, 1], 336),
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_{c[1]}x{c[2]}_n{c[6]}" for c in CASES])
def test_wide_tiles_match_oracle_and_256_column_tiles_bitwise(dev, case):
    from mixed_lora_projection_gb300 import _lib as L
    T, d_in, d_out, r, lens, ids, tn = case
    off = [0] + np.cumsum(lens).tolist()
    n_ad = max(ids)
    w = Workload("wide", 41, T, d_in, d_out, r, tuple(off), tuple(ids), n_adapters=max(n_ad, 1),
                 scales=(1.25, -0.75)[:max(n_ad, 1)])
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TILE_N, tn)
        assert _tile_n(ll, T, off, ids) == tn
        y = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_TILE_N, 256)
        y256 = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL
    assert torch.equal(y, y256)


@pytest.mark.parametrize("name", ["sweep_o", "sweep_down_multi"])
def test_model_choice_full_size(dev, name):
    # the 2,048-row o and down projections of the sweep: the model takes 288-column tiles (two
    # waves of SM pairs instead of three); sampled rows against the oracle, every row bitwise
    # against the same handle with wide tiles ruled out
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        assert _tile_n(ll, w.T, off, ids) == 288
        y = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_WIDE_TILES, 1)
        assert _tile_n(ll, w.T, off, ids) <= 256
        y_narrow = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=64)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], oracle_rows(inp, off, ids, rows)) <= TOL
    assert torch.equal(y, y_narrow)


def test_graph_replays_of_wide_tiles(dev):
    # a captured call with adapter rows (cooperative, ready flags) and one without, both on
    # 320-column tiles, replayed three times equal the eager calls
    from mixed_lora_projection_gb300 import _lib as L
    T = 700
    w = Workload("wide_graph", 42, T, 512, 1280, 32, (0, 300, T), (0, 1))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TILE_N, 320)
        cases = [([0, 300, T], [0, 1]), ([0, T], [0])]
        ref = [run(ll, inp, o, i).clone() for o, i in cases]
        outs = [torch.zeros_like(r) for r in ref]
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            for (o, i), y in zip(cases, outs):
                run(ll, inp, o, i, y=y)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        for y in outs:
            y.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for (o, i), y in zip(cases, outs):
                run(ll, inp, o, i, y=y)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert all(torch.equal(a, b) for a, b in zip(ref, outs))


def test_programmatic_dependent_launch_with_wide_tiles(dev):
    # a chain of base-row calls on 288-column tiles, each reading the previous call's Y, with
    # LORA_OPT_PDL (the first unit's W tiles requested before the dependency wait): equal to the
    # chain run without it
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    T = 600
    wa = Workload("widep_a", 43, T, 1024, 1536, 16, (0, T), (0,))
    wb = Workload("widep_b", 44, T, 1536, 1024, 16, (0, T), (0,))
    ia, ib = make_inputs(wa, dev), make_inputs(wb, dev)
    with LoraLinear(1024, 1536, 16, T, 4, 0) as ha, LoraLinear(1536, 1024, 16, T, 4, 0) as hb:
        for h in (ha, hb):
            h.set_option(L.OPT_TILE_N, 288)

        def chain(pdl):
            for h in (ha, hb):
                h.set_option(L.OPT_PDL, pdl)
            x, outs = ia.x, []
            for i in range(6):
                h, inp = (ha, ia) if i % 2 == 0 else (hb, ib)
                x = h.forward(x, [0, T], [0], inp.w, inp.a, inp.b, inp.scales)
                outs.append(x)
            return outs
        ref = [y.clone() for y in chain(0)]
        got = chain(1)
        torch.cuda.synchronize()
        assert ha.status() == 0 and hb.status() == 0
    assert all(torch.equal(a, b) for a, b in zip(ref, got))


def test_wait_that_runs_out_on_wide_tiles(dev):
    # the load warp never issues: both MMA warps' bounded waits run out, the call reports
    # LORA_ETIMEOUT, and the next call on the same handle is correct
    from mixed_lora_projection_gb300 import _lib as L
    T = 400
    off, ids = [0, 150, T], [1, 0]
    w = Workload("wide_stall", 45, T, 256, 640, 32, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TILE_N, 320)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        ll.set_option(L.OPT_DEBUG_STALL, 1)
        run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status(reset=True) == L.LORA_ETIMEOUT
        ll.set_option(L.OPT_DEBUG_STALL, 0)
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL


def test_options_that_rule_out_wide_tiles(dev):
    # single CTAs or K parts leave a forced wide width at 256 columns; widths past 512 or not a
    # multiple of 16 and an unknown LORA_OPT_WIDE_TILES value are rejected
    from mixed_lora_projection_gb300 import LoraError, _lib as L
    T = 600
    off, ids = [0, 200, T], [0, 1]
    w = Workload("wide_opts", 46, T, 6144, 512, 32, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y256 = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_TILE_N, 320)
        assert _tile_n(ll, T, off, ids) == 320
        ll.set_option(L.OPT_CLUSTER, 1)
        assert _tile_n(ll, T, off, ids) == 256
        ll.set_option(L.OPT_CLUSTER, 0)
        ll.set_option(L.OPT_K_SPLIT, 2)
        assert _tile_n(ll, T, off, ids) == 256
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
        for opt, v in ((L.OPT_TILE_N, 528), (L.OPT_TILE_N, 300), (L.OPT_WIDE_TILES, 2)):
            with pytest.raises(LoraError):
                ll.set_option(opt, v)
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL
    assert rel_err(y256, oracle_full(inp, off, ids)) <= TOL


@pytest.mark.parametrize("variant", ["raster1", "raster2", "raster3", "two_launch", "uploaded_list", "mma_group1",
                                     "max_ctas100"])
def test_wide_tiles_under_launch_options(dev, variant):
    # 320-column wide tiles under every launch option that touches their path (unit orders, the
    # shrink as its own launch, the work list uploaded instead of in the parameters, one stage per
    # MMA wait, a cap of 100 SMs) give the bits of 256-column tiles; the plain call matches the oracle
    from mixed_lora_projection_gb300 import _lib as L
    T = 1536
    off, ids = [0, 400, 1000, T], [0, 1, 2]
    w = Workload("wide_opts", 47, T, 640, 2000, 64, tuple(off), tuple(ids), n_adapters=2, scales=(0.5, 1.5))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TILE_N, 256)
        ref = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_TILE_N, 320)
        plain = run(ll, inp, off, ids).clone()
        if variant.startswith("raster"):
            ll.set_option(L.OPT_RASTER, int(variant[-1]))
            ll.set_option(L.OPT_RASTER_GROUP, 3)
        elif variant == "two_launch":
            ll.set_option(L.OPT_TWO_LAUNCH, 1)
        elif variant == "uploaded_list":
            ll.set_option(L.OPT_INLINE_WORK_LIST, 0)
        elif variant == "mma_group1":
            ll.set_option(L.OPT_MMA_GROUP, 1)
        else:
            ll.set_option(L.OPT_MAX_CTAS, 100)
        assert _tile_n(ll, T, off, ids) == 320
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(plain, ref)
    assert torch.equal(y, ref)
    assert rel_err(plain, oracle_full(inp, off, ids)) <= TOL


def test_two_wide_calls_side_by_side(dev):
    # the 2,048-row down projection as one call (288-column wide tiles on every SM pair), and as two
    # calls of 1,024 rows on two streams capped to 76 SMs each (wide tiles too): the same bits
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    w = WORKLOADS["sweep_down"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    y = torch.empty((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    main = torch.cuda.current_stream(dev)
    sa, sb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # rows 0..1023 and 1024..2047 in the batch's own segments
    cut = 1024
    oa, ia, ob, ib = [0], [], [0], []
    for k in range(len(ids)):
        lo, hi = off[k], off[k + 1]
        if lo < cut:
            oa.append(min(hi, cut)); ia.append(ids[k])
        if hi > cut:
            ob.append(hi - max(lo, cut) + ob[-1]); ib.append(ids[k])
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, 16, 0) as one, \
            LoraLinear(w.d_in, w.d_out, w.rank, cut, 16, 0) as ha, LoraLinear(w.d_in, w.d_out, w.rank, cut, 16, 0) as hb:
        assert _tile_n(one, w.T, off, ids) == 288
        ref = run(one, inp, off, ids).clone()
        for h in (ha, hb):
            h.set_option(L.OPT_MAX_CTAS, 76)
            h.set_option(L.OPT_TILE_N, 288)
        for _ in range(3):
            sa.wait_stream(main)
            sb.wait_stream(main)
            ha.forward(inp.x[:cut], oa, ia, inp.w, inp.a, inp.b, inp.scales, y=y[:cut], stream=sa)
            hb.forward(inp.x[cut:], ob, ib, inp.w, inp.a, inp.b, inp.scales, y=y[cut:], stream=sb)
            main.wait_stream(sa)
            main.wait_stream(sb)
        torch.cuda.synchronize()
        assert ha.status() == 0 and hb.status() == 0
    assert torch.equal(y, ref)
