"""bench.py on the CPU: the oracle arm (``--impl reference``) prints one JSON
line with the keys the line carries on the GPU arm, and under a multi-rank
launch only rank 0 does the work and prints; the algorithmic bytes the GPU
arm's roofline objects divide by time match counts written out by hand."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
       "--warmup", "3"]


def _run(extra_env, extra_args=()):
    env = dict(os.environ, **extra_env)
    return subprocess.run(CMD + list(extra_args), cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, ["--gpus", "2"])
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_gpus_flag_launches_that_many_replicas():
    """``--gpus 2`` without a launcher starts two ranks itself; rank 0 alone
    prints one line, which reports both."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run(CMD + ["--gpus", "2"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_gpus_flag_must_match_the_launch():
    r = _run({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})  # --gpus defaults to 1
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_roofline_numerators_match_hand_counts():
    """The algorithmic bytes the bench divides by time, against counts written
    out by hand from the workload shapes."""
    sys.path.insert(0, ROOT)
    import workloads as W
    b = _bench_module()
    # scheduler-step prefill: T = 4096, H = 32, d = 128, bf16 in, fp32 state,
    # 8 live sequences, checkpoints every 256 tokens (6+2+0+0+0+1+3+1 = 13)
    w = W.SCHED
    d = W.make_prefill(w)
    T, H, dd = 4096, 32, 128
    state = dd * dd * 4
    expect = (4 * T * H * dd * 2          # q, k, g, v
              + T * H * 2                 # beta
              + T * H * dd * 2            # out
              + T * H * dd * 2 + dd * 2   # gate, norm weight
              + 2 * 8 * H * state         # state read + write
              + 13 * H * state)           # checkpoints
    assert expect == 262_406_400
    assert b.prefill_algorithmic(w, d)[0] == expect
    # decode: 256 sequences, fp32 states read and written, 641 bf16 values per
    # (sequence, head) of q, k, g, v, beta, out, the gate, the weight, indices
    dw = W.DECODE
    expect = 2 * 256 * H * state + 256 * H * (3 * dd + dd + 1 + dd) * 2 + 256 * H * dd * 2 + dd * 2 + 256 * 4
    assert expect == 1_086_342_400
    assert b.decode_algorithmic(dw)[0] == expect
    # verification of 4 draft tokens: state read, 4 states written, inputs and
    # outputs of 4 tokens, and the commit of every sequence with a_i > 0
    dr = W.make_decode_draft(dw, 4)
    n_acc = int((dr["num_accepted"] > 0).sum())
    expect = (256 * H * state + 4 * 256 * H * state + 4 * 256 * H * (3 * dd + dd + 1 + dd) * 2
              + 4 * 256 * H * dd * 2 + dd * 2 + 2 * n_acc * H * state + 256 * 8)
    assert b.spec_algorithmic(dw, 4, dr["num_accepted"]) == expect
    # convolution over 12288 channels, width 4: x read and y written, taps and
    # bias, 8 caches of 3 rows read and written
    C = 3 * H * dd
    expect = 2 * T * C * 2 + C * 5 * 2 + 2 * 8 * 3 * C * 2
    assert expect == 202_629_120
    assert b.conv_algorithmic(w, C, 4) == expect
    # one 4096-token call of the long prompt: bf16 inputs, no gate, bf16 state
    # read and written once, 16 bf16 checkpoints
    lw = W.LONGPROMPT.replace(seqlens=(4096,))
    bstate = dd * dd * 2
    expect = 4 * T * H * dd * 2 + T * H * 2 + T * H * dd * 2 + 2 * H * bstate + 16 * H * bstate
    assert expect == 186_908_672
    assert b.prefill_algorithmic(lw, {"cu_seqlens": W.cu_from_lengths([4096])})[0] == expect
    # the scheduler step with the width-4 convolution fused in: the prefill's
    # bytes (the packed projection x replaces q, k, v, the same size), taps and
    # bias of 3 x 32 x 128 channels, 8 convolution caches of 3 rows read and
    # written
    expect = 262_406_400 + C * 5 * 2 + 2 * 8 * 3 * C * 2
    assert expect == 263_708_928
    assert b.prefill_conv_algorithmic(w, d, 4)[0] == expect


def test_prefill_flop_count_matches_hand_count():
    """Full 64-row chunks with d = 128: 2 (KK^T, QK^T lower triangles) x
    2 x 2080 x 128, the triangular inverse 64^3 / 3, W and U0 2 x 2080 x 256,
    the three state products 6 x 64 x 128 x 128, A_qk U 2 x 2080 x 128 and the
    decay scaling 4 x 64 x 128 FLOPs per chunk-head."""
    sys.path.insert(0, ROOT)
    import workloads as W
    b = _bench_module()
    per_chunk = (4 * 2080 * 128 + 64 ** 3 / 3 + 2 * 2080 * 256 + 6 * 64 * 128 * 128
                 + 2 * 2080 * 128 + 4 * 64 * 128)
    w = W.SCHED.replace(seqlens=(128, 64), H=2, num_slots=4, slot_range=None)
    d = W.make_prefill(w)
    assert abs(b.prefill_algorithmic(w, d)[1] - 3 * 2 * per_chunk) < 1e-3
