"""The roofline arithmetic of bench.py against the per-workload figures worked out by hand from
the workload definitions (bytes moved and dual-form FLOPs per launch or step).

Per head-token: TTT-Linear 6 d^2 + 2 (b + 1) d FLOPs (Q W0, K W0 and the K^T E update, plus the
causal scores and A E); TTT-MLP 14 d h + 2 (b + 1)(d + h).  Bytes: Q, K, V, Z in the I/O dtype and eta
in fp32 per head-token, the fp32 state read and written once per head (prefill) or per step (decode).
"""
import bench


def test_linear_prefill_headline():
    # B=8 H=12 d=64 T=2048 b=16: 196,608 head-tokens x 26,752 FLOPs; 101.45 MB of Q/K/V/Z/eta + 3.15 MB of state
    assert bench.linear_flops(8, 12, 2048, 64, 16) == 196_608 * 26_752
    assert bench.linear_bytes(8, 12, 2048, 64) == 104_595_456


def test_mlp_prefill():
    # hidden 256: 196,608 head-tokens x 240,256 FLOPs (47.24 GFLOP); + 25.17 MB of W1, W2 in and out
    assert bench.mlp_flops(8, 12, 2048, 64, 256, 16) == 196_608 * 240_256
    assert bench.mlp_bytes(8, 12, 2048, 64, 256) == 126_615_552


def test_long_context():
    # B=1 H=16 d=128 T=32768: 524,288 head-tokens x (98,304 + 256 (b + 1)) FLOPs; 541.07 MB
    for b, per_token in ((16, 102_656), (64, 114_944), (512, 229_632)):
        assert bench.linear_flops(1, 16, 32768, 128, b) == 524_288 * per_token
    assert bench.linear_bytes(1, 16, 32768, 128) == 541_065_216


def test_decode_step():
    # B=256 H=12 d=64: the 100.66 MB fp32 state read and written, 1.59 MB of q, k, v, z, eta
    assert bench.decode_bytes(256, 12, 64) == 102_248_448


def test_mlp_decode_step():
    # B=64 H=12 d=64 hidden=256: W1 and W2 (2 x 64 KB fp32 per head) read and written, q, k, v, z, eta
    assert bench.mlp_decode_bytes(64, 12, 64, 256) == 201_722_880


def test_backward_headline():
    # Q, K, V, dZ read and dQ, dK, dV written (7 x 25.17 MB), eta read and deta written, one bf16 state per
    # 16-token block read (100.66 MB), dW_T read and dW0 written (2 x 1.57 MB)
    assert bench.backward_bytes(8, 12, 2048, 64, 16) == 281_542_656
    # 14 d^2 + 5 (b + 1) d = 62,784 FLOPs per head-token: 12.34 GFLOP
    assert bench.backward_flops(8, 12, 2048, 64, 16) == 12_343_836_672
