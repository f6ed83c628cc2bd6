"""Host-side checks of bench.py's bookkeeping (no GPU): the algorithmic bytes
behind every roofline figure are the bytes of the operands the bench builds,
and the DRAM traffic it reports is tied to the kernel sources it was
captured from and to the profile summary that records it."""
import importlib.util
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_are_the_operands(bench):
    # every step operation at a reduced size: the bytes the roofline counts
    # are those of the tensors the kernel reads (the combine's scalar scale
    # is a launch argument, not a stream) plus those it writes
    for name, _, spec in bench.op_specs():
        small = dict(spec)
        small["rows"] = min(spec["rows"], 48)
        if "cols" in small:
            small["cols"] = min(spec["cols"], 72)
        ins = bench.make_inputs(small, "cpu")
        outs = bench.make_outputs(small, ins, "cpu")
        streamed = ins[:3] if small["kind"] == "combine" else ins
        bi, bo = bench.algorithmic_bytes(small)
        assert bi == sum(t.numel() * t.element_size() for t in streamed), name
        assert bo == sum(t.numel() * t.element_size() for t in outs), name


def test_source_hash_ignores_comments_only(bench, tmp_path, monkeypatch):
    d = tmp_path / "cluster_reductions_gb300" / "csrc"
    d.mkdir(parents=True)
    f = d / "k.cu"
    f.write_text("// a kernel\n__global__ void k(float *x) { x[0] = 1.0f; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_src_sha(["k.cu"])
    f.write_text("/* the same kernel,\n   re-commented */\n__global__ void k(float *x) {\n"
                 "  x[0] = 1.0f;  // store\n}\n")
    assert bench.kernel_src_sha(["k.cu"]) == h0
    f.write_text("__global__ void k(float *x) { x[0] = 2.0f; }\n")
    assert bench.kernel_src_sha(["k.cu"]) != h0


def test_traffic_dropped_when_the_kernel_changes(bench, tmp_path, monkeypatch):
    d = tmp_path / "cluster_reductions_gb300" / "csrc"
    d.mkdir(parents=True)
    (d / "k.cu").write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_src_sha(["k.cu"])
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {
        "op": {"bytes": 123, "src": ["k.cu"], "src_sha": sha, "profile": "p.md"}})
    assert bench.ncu_traffic("op")["bytes"] == 123
    assert bench.ncu_traffic("other") is None
    (d / "k.cu").write_text("__global__ void k() { __syncthreads(); }\n")
    assert bench.ncu_traffic("op") is None


def test_traffic_figures_match_their_profiles(bench):
    # each recorded per-launch traffic figure is the one its profile summary
    # states for a full-size launch (MB, one decimal); a summary that was
    # re-captured states its latest figure last
    for name, tr in bench.NCU_TRAFFIC.items():
        path = os.path.join(ROOT, tr["profile"])
        assert os.path.exists(path), (name, path)
        text = open(path).read()
        m = re.findall(r"per full-size launch \(x[0-9.]+ units\): ([0-9.]+) MB", text)
        assert m, (name, path)
        assert abs(float(m[-1]) - tr["bytes"] / 1e6) <= 0.05 + 1e-9, (name, m[-1])
        assert name in dict((n, 0) for n, _, _ in bench.op_specs()), name
