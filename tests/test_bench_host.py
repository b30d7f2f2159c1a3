"""Host logic of the benchmark's multi-rank mode, on CPU with gloo: each rank
runs its own replica, the line reports the sum of the ranks' bytes over the
slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    dev = torch.device("cpu")
    region_ms = [10.0, 12.5][rank]
    step_bytes = [1000.0, 1000.0][rank]
    out[rank] = (bench.reduce_max(region_ms, world, dev), bench.reduce_sum(step_bytes, world, dev),
                 bench.dist_env())
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
        got = dict(out)
    for rank in range(world):
        mx, total, env = got[rank]
        assert mx == 12.5          # slowest rank's time
        assert total == 2000.0     # all ranks' bytes
        assert env == (rank, world, rank)


def test_single_rank_reductions_are_identity():
    assert bench.reduce_max(3.0, 1, None) == 3.0
    assert bench.reduce_sum(4.0, 1, None) == 4.0


def test_reference_arm_under_two_ranks_prints_one_line():
    """torchrun with two CPU ranks: rank 0 times the oracle and prints one
    JSON line with the arm's fields, rank 1 exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1", "--ref-budget-s", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == bench.STEP_CONFIG["workload"]


def _stitch(outs):
    """The oracle's range outputs of each call joined into whole arrays: a
    stand-in for the GPU outputs read back from the timed buffers."""
    import numpy as np
    return [{k: np.concatenate([r[k] for _, r in o]) for k in o[0][1] if k != "bad"}
            for o in outs]


def test_parity_gate_passes_on_oracle_outputs_and_flags_planted_errors():
    """The bench's parity gate on the first 1 % of every step call's rows:
    the oracle's own outputs pass; one wrong bit in residual_out or a
    gathered row, a normalised value off by 0.01, a nonzero pad row or an
    fp32 GELU value off by 3e-5 relative each fail their call."""
    import numpy as np
    calls = bench.build_calls(gpu=False)
    _, _, outs = bench.oracle_step(calls, 2, 0.01)
    good = bench.parity_gate(calls, _stitch(outs), outs, 2)
    assert good["pass"] and "failures" not in good
    assert good["elements"] == sum(v.size for g in _stitch(outs) for v in g.values())
    assert good["bitwise"] > 0 and good["ln"]["n"] > 0
    assert good["gelu_f32"]["n"] > 0 and good["gelu_f16"]["n"] > 0
    labels = [c.label for c in calls]
    bad = _stitch(outs)
    j = labels.index("residual_add_ln_fwd [131040,192]")
    bad[j]["r"].view(np.uint16)[7, 3] ^= 1
    j = labels.index("window_gather [32760,384]->34560")
    bad[j]["dst"].view(np.uint16)[10, 5] ^= 0x8000
    j = labels.index("norm_gather [131040,192]->138240")
    row = int(np.nonzero(bench._oracle_map(bench.synth.STAGE_192)[:bad[j]["dst"].shape[0]] >= 0)[0][0])
    bad[j]["dst"][row, 9] += np.float16(0.01)
    j = labels.index("norm_gather [32760,384]->34560")
    pads = np.nonzero(bench._oracle_map(bench.synth.STAGE_384)[:bad[j]["dst"].shape[0]] < 0)[0]
    if pads.size:  # the first 1 % of the C = 384 map holds pad rows
        bad[j]["dst"][pads[0], 0] = np.float16(1.0)
    j = labels.index("bias_gelu_tanh fp32 [131040,768]")
    bad[j]["y"][5, 5] *= np.float32(1 + 3e-5)
    got = bench.parity_gate(calls, bad, outs, 2)
    assert not got["pass"]
    failed = {f.split(":")[0] for f in got["failures"]}
    want = {"residual_add_ln_fwd [131040,192]", "window_gather [32760,384]->34560",
            "norm_gather [131040,192]->138240", "bias_gelu_tanh fp32 [131040,768]"}
    if pads.size:
        want.add("norm_gather [32760,384]->34560")
    assert failed == want


def test_reference_arm_never_loads_the_cuda_library():
    """The reference arm builds its index maps with the oracle, so a run of
    it leaves libwgs.so unloaded."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys, json; sys.argv=['bench.py','--impl','reference','--steps','1','--warmup',"
            "'1','--ref-budget-s','1']; import bench; bench.main(sys.argv[1:]); "
            "maps=open('/proc/self/maps').read(); print(json.dumps({'wgs': 'libwgs.so' in maps}))")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert json.loads(lines[-1]) == {"wgs": False}
    ref = json.loads(lines[0])
    assert ref["impl"] == "reference" and ref["cpu_baseline"]["host_cores"] >= 1


def test_cpu_legs_skip_calls_without_an_oracle_leg():
    """A call without an oracle leg (a --only subset can hold one) leaves the
    others' GPU outputs matched to their own calls."""
    calls = [c for c in bench.build_calls(gpu=False) if c.workload == "[32760,384]"]
    assert [c.name for c in calls] == ["ln_fwd", "residual_add_ln_fwd"]
    _, _, outs = bench.oracle_step(calls, 2, 1.0)
    gpu = _stitch(outs)
    extra = bench.Call("no_leg", "x", 0, {}, {}, None, None, 0)
    base, parity = bench.cpu_legs([calls[0], extra, calls[1]], [gpu[0], None, gpu[1]],
                                  want_baseline=False, want_parity=True)
    assert base is None
    assert parity["pass"], parity.get("failures")
    assert parity["elements"] == sum(v.size for g in gpu for v in g.values())
