"""bench.py host logic that needs no GPU: the algorithmic byte models (the
numerators of its roofline fractions), pinned per request at 16 heads x 128
to the figures written out from the tensors each call must read or write
once; and the --impl reference arm, which times the FP64 oracle on the host
cores and prints the same JSON line contract."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STATE = 16 * 128 * 128 * 4             # one request's FP32 state, 16 heads
TOKEN = 12288 + 4096 + 32 + 4096       # packed q/k/v row, gate input, beta, o (BF16)
RING = 16 * (3 * 128 + 4) * 4          # replayed ring records of one token


def test_token_io():
    assert bench.token_io_bytes() == TOKEN == 20512


def test_per_request_models():
    assert bench.decode_bytes(1) == 2 * STATE + TOKEN == 2117664
    assert bench.verify_bytes(1, 6) == STATE + 6 * STATE + 6 * TOKEN == 7463104
    assert bench.commit_bytes(1) == 2 * STATE
    assert bench.verify_replay_bytes(1, 6) == STATE + 6 * TOKEN + 6 * RING == 1320640
    # a request that accepted draft token 2 replays 3 ring records; -1 moves nothing
    assert bench.commit_replay_bytes([2, -1], 6) == 2 * STATE + 3 * RING


def test_models_scale_with_requests():
    assert bench.decode_bytes(48) == 48 * bench.decode_bytes(1)
    assert bench.verify_bytes(16, 6) == 16 * bench.verify_bytes(1, 6)


def test_transform_input_bytes():
    # q, k, v and the gate input (BF16, T x 16 x 128 each) and beta (T x 16)
    assert bench.transform_bytes(4096) == 4 * 4096 * 16 * 128 * 2 + 4096 * 16 * 2 == 67239936


def _reference(env=None):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return [json.loads(line) for line in out.stdout.splitlines() if line.startswith("{")]


def test_reference_arm_prints_the_contract_line():
    (j,) = _reference()
    assert j["impl"] == "reference"
    assert j["metric"] == bench.METRIC and j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert (j["n_gpus"], j["steps"], j["warmup"]) == (1, 1, 3)
    assert j["value"] > 0 and j["ms_per_step"] > 0
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"] and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    assert _reference(env) == []
