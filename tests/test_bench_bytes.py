"""The algorithmic byte counts behind the benchmark's roofline fractions,
against the Qwen3-8B shape worked out by hand."""
import bench
from invariant_deterministic_gb300 import model as M


def test_gemm_bytes_is_operands_plus_output():
    # 2 bytes per bf16 element of A [M][K], W [N][K] and C [M][N]
    assert bench.gemm_bytes(16, 6144, 4096) == 2 * (16 * 4096 + 6144 * 4096 + 16 * 6144)
    assert bench.gemm_bytes(1, 151936, 4096, out_bytes=4) == 2 * (4096 + 151936 * 4096) + 4 * 151936


def test_decode_step_bytes_of_the_8b_shape():
    s = M.QWEN3_8B
    # per layer: QKV 6144 x 4096, O 4096 x 4096, gate+up 2 x 12288 x 4096,
    # down 4096 x 12288 = 192.94 M parameters, plus two norm gains of 4096
    per_layer = (6144 * 4096 + 4096 * 4096 + 2 * 12288 * 4096 + 4096 * 12288) * 2 + 2 * 4096 * 2
    assert per_layer == 385_892_352
    lm_head = 151936 * 4096 * 2
    kv_per_position = 8 * 128 * 2 * 2 * 36          # K and V, 8 heads of 128, bf16, 36 layers
    assert kv_per_position == 147_456
    lens = [100, 2000]
    got = bench.step_bytes(s, 2, lens)
    weights = 36 * per_layer + lm_head + 2 * 4096 * 2 + 4096 * 2   # + embedding rows, final norm gain
    kv = sum(l + 1 for l in lens) * kv_per_position + 2 * kv_per_position   # read, and the new rows written
    logits = 2 * 151936 * 4 * 2                      # fp32, written and read
    assert got == weights + kv + logits
    # about 15.14 GB of weights per step
    assert abs((36 * per_layer + lm_head) / 1e9 - 15.14) < 0.01
    # one more cached position costs every request exactly its K/V row
    assert bench.step_bytes(s, 2, [101, 2000]) - got == kv_per_position
