"""Fixtures under tests/golden/: the pages' printed parameters (with the
values the implementation's readings derive from them) and the oracle's
regression values (written by tests/golden/make_golden.py from oracle/)."""
import json
import os

from oracle import oracle as O
from streaming_diffusion_stream_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_pages_t_index_list_maps_to_the_stated_timesteps():
    g = load("pages_parameters.json")["t_index_list"]
    w = W.get_config("c1_tiny", t_index=g["value"])
    assert [O.slot_timestep(w, i) for i in range(len(g["value"]))] == g["derived_timesteps"]


def test_pages_r_cfg_table_is_self_consistent():
    g = load("pages_parameters.json")["r_cfg_speedup_5_steps"]["value"]
    assert round(g["cfg_ms"] / g["self_negative_ms"], 2) == g["self_speedup"]


def close(got, want, path="") -> None:
    """Recursive comparison: integers exactly, floats to 1e-13 relative."""
    if isinstance(want, dict):
        assert got.keys() == want.keys(), path
        for k in want:
            close(got[k], want[k], f"{path}/{k}")
    elif isinstance(want, list):
        assert isinstance(got, list) and len(got) == len(want), path
        for i, (g, x) in enumerate(zip(got, want)):
            close(g, x, f"{path}[{i}]")
    elif isinstance(want, float):
        assert abs(got - want) <= 1e-13 * max(1.0, abs(want)), (path, got, want)
    else:
        assert got == want, (path, got, want)


def test_oracle_matches_its_regression_fixture():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    close(json.loads(json.dumps(mg.compute())), load("oracle_regression.json"))
