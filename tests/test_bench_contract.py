"""The benchmark's reference arm and its JSON line, on the host (no GPU).

The reference arm times the CPU oracle through the same workload, metric and
units as the GPU arm; the driver divides the two lines' values, so their keys,
units and direction must agree.
"""
import json

import pytest

import bench

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
            "impl", "cpu_baseline", "e2e"}


def _run(capsys, argv):
    assert bench.main(argv) == 0
    out = capsys.readouterr().out.strip().splitlines()
    return out


def test_reference_arm_line(capsys, monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    out = _run(capsys, ["--impl", "reference", "--config", "0", "--steps", "2", "--warmup", "1"])
    assert len(out) == 1, out
    d = json.loads(out[0])
    assert REQUIRED <= set(d)
    assert d["metric"] == bench.METRIC
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.make_workload(0).name
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_only_rank0_prints(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert _run(capsys, ["--impl", "reference", "--config", "0", "--steps", "1",
                         "--warmup", "0"]) == []


@pytest.mark.parametrize("config", [0, 1, 2, 3, 4])
def test_replicas_have_the_same_shapes_and_their_own_data(config):
    """Weak scaling: every rank runs the same workload shape with its own seed."""
    a, b = bench.make_workload(config, 0), bench.make_workload(config, 1)
    assert a.name == b.name and a.layers == b.layers and a.head_dim == b.head_dim
    assert len(a.steps) == len(b.steps)
    sa, sb = a.steps[-1], b.steps[-1]
    assert sa.q[0].shape == sb.q[0].shape
    assert sa.k_new.shape[1:] == sb.k_new.shape[1:]
    assert not (sa.q[0] == sb.q[0]).all()


def test_reference_config_matches_the_gpu_arm(capsys, monkeypatch):
    """Both arms print the same `config` for the same workload, so the driver can pair them."""
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    out = _run(capsys, ["--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "0"])
    d = json.loads(out[0])
    wl = bench.make_workload(0)
    st = wl.steps[-1]
    assert d["config"] == bench.workload_config(wl, st, bench.accounting(wl, st), 1)


def test_kernel_hash_ignores_comments_only():
    """The traffic figures stay attached to the kernel's code: a comment or blank-line
    edit keeps the hash, any code edit changes it."""
    import bench
    src = "int a = 1;  // one\n/* block\n comment */\n\nint b = 2;\n"
    assert bench._code_only(src) == bench._code_only("int a = 1;\n// other words\nint b = 2;\n")
    assert bench._code_only(src) != bench._code_only("int a = 1;\nint b = 3;\n")
