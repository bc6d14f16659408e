"""Geometry printed on the source pages, against the workloads the tests and bench use."""
import os

from mixed_lora_projection_gb300.synth import WORKLOADS, SWEEP_PROJECTIONS

HERE = os.path.dirname(os.path.abspath(__file__))


def _read():
    vals = {}
    with open(os.path.join(HERE, "golden", "adapter_geometry.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_page_geometry_is_self_consistent():
    g = _read()
    # the parameter count is rank x sum over changed matrices of (d_in + d_out)
    assert g["adapter_parameters"] % g["rank"] == 0
    assert g["layers_last_adapted"] - g["layers_first_adapted"] + 1 == 24
    # bf16: two bytes per parameter, printed to one decimal in GiB
    assert abs(g["adapter_parameters"] * 2 / 2 ** 30 - g["adapter_bf16_gib"]) < 0.05


def test_workloads_use_the_page_geometry():
    g = _read()
    for name in ("prefill_16k", "mixed_batch", "mixed_decode", "prefill_32k"):
        w = WORKLOADS[name]
        assert w.rank == g["rank"]
        assert g["hidden"] in (w.d_in, w.d_out)
    for proj, d_in, d_out in SWEEP_PROJECTIONS:
        assert g["hidden"] in (d_in, d_out)
