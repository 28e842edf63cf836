"""The algorithmic byte and flop counts behind the bench line's roofline fractions, against closed
forms worked out by hand for the bench workloads (d_k = d_v = 128, bf16 token tensors, fp32 state)."""
import bench
import synth


def test_chunk_bytes_of_the_prefill_workload():
    wl = synth.WORKLOADS["prefill32k_decode"]
    # per token: q, k on 16 key heads + g, b (d_k) and v, w (d_v) on 32 value heads + o, bf16
    per_token = (2 * 16 * 128 + 32 * (128 + 128 + 128 + 128) + 32 * 128) * 2
    assert per_token == 49_152
    final_state = 2 * 32 * 128 * 128 * 4
    assert bench.chunk_bytes(wl) == 2 * 32768 * per_token + final_state == 3_225_419_776


def test_chunk_flops_are_triangle_aware():
    wl = synth.WORKLOADS["prefill32k_decode"]
    # per (head, token): the C x C products counted once per pair (C (3 d_k + 2 d_v)) + 6 d_k d_v
    per = 64 * (3 * 128 + 2 * 128) + 6 * 128 * 128
    assert per == 139_264
    assert bench.chunk_flops(wl) == 2 * 32768 * 32 * per == 292_057_776_128


def test_decode_step_bytes_of_the_serving_shape():
    # fp32 state read and written once, one token's inputs and output
    state = 2 * 64 * 48 * 128 * 128 * 4
    tokens = 64 * (2 * 16 * 128 + 48 * (2 * 128 + 2 * 128)) * 2 + 64 * 48 * 128 * 2
    assert bench.decode_step_bytes(64, 16, 48, 128, 128) == state + tokens == 407_109_632


def test_backward_flops():
    assert bench.backward_flops(2 * 32768, 32, 128) == 26 * 128 * 128 * 65536 * 32 == 893_353_197_568
