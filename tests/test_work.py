"""Work accounting: brute-force pair counts and the pages' ~6x reduction claim."""
import pytest

from hybrid_sliding_window_02_b300 import work


@pytest.mark.parametrize("T,W", [(0, 4), (1, 1), (5, 1), (9, 4), (16, 16), (16, 40), (100, 7)])
def test_window_pairs_brute(T, W):
    n = sum(1 for i in range(T) for j in range(T) if j <= i and i - j < W)
    assert work.window_pairs(T, W) == n


def test_decode_bytes_full_size():
    # 256 sequences, Hq=64, Hkv=8, D=128, W=128 bf16 rings, fp32 out + lse
    assert work.decode_bytes(256, 64, 8, 128, 128, 2) == 146_868_480


def test_prefill_work_full_size():
    assert work.prefill_flops(4, 8192, 64, 128, 128) == 4 * 128 * 4 * 64 * (
        128 * 129 // 2 + (8192 - 128) * 128)
    assert work.prefill_bytes(4, 8192, 64, 8, 128, 2) == (
        4 * 8192 * 80 * 128 * 2 + 256 + 4 * 8192 * 64 * 128 * 4 + 4 * 64 * 8192 * 4)


def test_hybrid_reduction_about_six():
    # "近6倍" (nearly 6x) KV-cache and attention-FLOP reduction at 5:1, W=128
    f32k, kv32k = work.hybrid_reduction(32768)
    f256k, kv256k = work.hybrid_reduction(262144)
    assert 5.7 < f32k < 6.0 and 5.8 < kv32k < 6.0
    assert 5.9 < f256k < 6.0 and 5.9 < kv256k < 6.0
    assert f256k > f32k and kv256k > kv32k          # tends to 6 as T grows
    f, kv = work.hybrid_reduction(10 ** 9)
    assert abs(f - 6) < 1e-3 and abs(kv - 6) < 1e-3


def test_verify_work_counts():
    from hybrid_sliding_window_02_b300 import work
    # one drafted token is a decode against the ring plus itself: same bytes
    # as decode except the new key/value rows instead of nothing
    B, Hq, Hkv, D, W = 256, 64, 8, 128, 128
    assert work.verify_bytes(B, 1, Hq, Hkv, D, W, 2) == (
        work.decode_bytes(B, Hq, Hkv, D, W, 2) + 2 * B * Hkv * D * 2)
    assert work.verify_pairs(4, 128, 1000) == 4 * 128
    assert work.verify_pairs(3, 128, 0) == 1 + 2 + 3


def test_hybrid_reduction_seven_to_one():
    # the 7:1 schedule of the later models, stated as a 7x cut in attention
    # FLOPs and KV cache ("MiMo-V2.5" ICML 2026 talk write-up, intro and 02):
    # the closed form is about 7.6x / 7.8x at 32K and tends to 8x with length
    from hybrid_sliding_window_02_b300 import work
    flop, kv = work.hybrid_reduction(32768, 128, 7, 1)
    assert 7.0 <= flop < 8.0 and 7.0 <= kv < 8.0
    flop_long, kv_long = work.hybrid_reduction(262144, 128, 7, 1)
    assert flop < flop_long < 8.0 and kv < kv_long < 8.0


def test_append_byte_counts():
    from hybrid_sliding_window_02_b300 import work
    # 256 sequences, 8 kv heads, D = 128, bf16: k and v of the new token
    # (2 x 512 KB) read and written once, pos 2 KB; the fused step adds q
    # (4 MB) read and its rotated copy written
    assert work.append_bytes(256, 8, 128, 2) == 4 * 524_288 + 2048
    assert work.rope_append_bytes(256, 64, 8, 128, 2) == (
        work.append_bytes(256, 8, 128, 2) + 2 * 4_194_304)


def test_rope_byte_count():
    from hybrid_sliding_window_02_b300 import work
    # q of the headline prefill (B4 T8192 Hq64 D128 bf16, 536,870,912 B) read
    # and written, plus 4 int64 start positions
    assert work.rope_bytes(4, 8192, 64, 128, 2) == 2 * 536_870_912 + 32
