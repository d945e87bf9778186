"""The byte models the bench divides by, checked on the CPU against the
figures the workload definitions give (one read of every source row, one
write of r and of the weights)."""
import bench


def test_single_layer_algorithmic_bytes():
    # T * (S d 2 + d 2 + S 4): bf16 sources and r, fp32 weights
    assert bench.algorithmic_bytes(4096, 7168, 9) == 587_350_016             # the bench step
    assert bench.algorithmic_bytes(131072, 7168, 9) == 18_795_200_512        # long context
    assert bench.algorithmic_bytes(2048, 7168, 94) == 2_789_982_208          # Full AttnRes, 94 sources
    # per token: 9 rows of 14,336 B, r 14,336 B, 9 weights of 4 B
    assert bench.algorithmic_bytes(1, 7168, 9) == 9 * 14_336 + 14_336 + 36
    # the small fp32 layer: 4 sources and r of 256 fp32, 4 weights, 64 tokens
    assert 64 * (4 * 256 * 4 + 256 * 4 + 4 * 4) == 328_704
    assert bench.algorithmic_bytes(64, 256, 4, esz=4) == 328_704


def test_roofline_time_of_the_bench_step():
    # at the measured copy bandwidth of 6,786.9 GB/s the step takes 86.5 us:
    # the figure the fraction is taken against
    t_us = bench.algorithmic_bytes(4096, 7168, 9) / 6786.9e9 * 1e6
    assert abs(t_us - 86.54) < 0.01
