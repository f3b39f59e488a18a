"""CPU checks of bench.py's host arithmetic: the algorithmic flops and bytes
that the roofline fractions divide by, against closed forms worked out by
hand for the five workloads (no GPU)."""
import os

import pytest

import bench
from mixture_experts_ffn_02_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# forward flop = 2 per multiply-add x 3 products (gate, up, down) x d x
# (k H per real token for the routed slots + n_s H_s for the shared expert),
# expanded by hand for each workload
FWD_FLOP = {
    1: 2 * 256 * 3 * 64 * (2 * 128 + 1 * 128),          # tiny: 0.0377 GFLOP
    2: 2 * 32768 * 3 * 1536 * (2 * 3072 + 1 * 3072),    # KochiLLM: 2783.1 GFLOP
    3: 2 * 60293 * 3 * 512 * (2 * 768),                 # packed, real tokens: 284.5 GFLOP
    4: 2 * 16384 * 3 * 2048 * (6 * 1408 + 2 * 1408),    # 64 experts top-6: 2267.7 GFLOP
    5: 2 * 32768 * 3 * 1024 * (8 * 768),                # 128 experts top-8: 1237.0 GFLOP
}


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_gemm_flops_closed_form(cfg):
    s = synth.shape(cfg)
    routed, shared = bench.gemm_flops(s)
    Tr = s.T_real if s.T_real is not None else s.T
    assert routed == 2 * Tr * s.k * 3 * s.d * s.H
    assert shared == 2 * Tr * 3 * s.d * s.n_shared * s.H_shared
    assert routed + shared == FWD_FLOP[cfg]


def test_hbm_bytes_closed_forms():
    """KochiLLM shape (T = 32768, d = 1536, k = 2, no PAD): the permute reads
    x once (100.7 MB), writes 65536 rows of x_perm (201.3 MB) and moves
    4 bytes per topk entry in, per perm entry and per inv entry out; the
    packed shape counts real tokens only for the row traffic."""
    s = synth.shape(2)
    b = bench.hbm_bytes(s)
    T, d, k = 32768, 1536, 2
    assert b["permute"] == T * d * 2 + T * k * d * 2 + 3 * T * k * 4 == 302776320
    assert b["router_route"] == T * d * 2 + d * 4 * 4 + T * 4 * 4 + T * k * 8
    p = synth.shape(3)
    bp = bench.hbm_bytes(p)
    Tr, M = 60293, 60293 * 2
    assert bp["permute"] == Tr * 512 * 2 + M * 512 * 2 + 65536 * 2 * 4 + M * 4 + 65536 * 2 * 4
    # out_perm bf16 in, no shared expert, inv + gates in, y (bf16, all positions) out
    assert bp["combine"] == M * 512 * 2 + 65536 * 2 * 8 + 65536 * 512 * 2


def test_aggregate_single_rank():
    ms, v = bench.aggregate_ranks(200.0, 32768, 5, 1)
    assert ms == 200.0 and v == pytest.approx(32768 * 5 / 0.2)


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference runs the fp64 oracle (no GPU) and prints one
    JSON line with the same metric, the impl tag, its CPU baseline and an
    e2e block with no host copies."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "1", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["nproc"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_launches_per_step_count_the_kernels_of_each_path(monkeypatch):
    """The gpu_launches claim: kernels of this library per step, counted by
    hand from the launch lists of each path.  E <= 16: the streamed router
    (zeroing kernel + router, 2), the permute (3), gate/up and down, the
    shared expert's two GEMMs with the combine folded in (or the combine
    kernel), and the backward (combine backward, dH, dX, two dW, the shared
    expert's four GEMMs or the dx gather, and the router's dW_r and its split
    sum).  E a multiple of 32: the logits SGEMM and the route kernel, and the
    router's five-launch tensor-core backward."""
    monkeypatch.delenv("MOE_ROUTER_STREAM", raising=False)
    expect = {1: (9, 20), 2: (9, 20), 3: (8, 16), 4: (9, 23), 5: (8, 19)}
    for c, (fwd, both) in expect.items():
        s = synth.shape(c)
        assert bench.launches_per_step(s, True) == fwd, c
        assert bench.launches_per_step(s, False) == both, c
    monkeypatch.setenv("MOE_ROUTER_STREAM", "0")              # one-kernel fused router
    assert bench.launches_per_step(synth.shape(2), False) == 19
