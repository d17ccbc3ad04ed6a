"""bench.py's algorithmic byte models (the numerators of its roofline
fractions), pinned per request at 16 heads x 128 to the figures written out
from the tensors each call must read or write once."""
import bench

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
