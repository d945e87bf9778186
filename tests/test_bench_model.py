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


def _simulated_stack_bytes(T, d, esz, L, B):
    # the stack's state followed layer by layer: the stored rows (h_0 and the
    # closed blocks) and whether the current block has a partial sum; each
    # step reads every stored row, the partial and F once and writes the
    # folded row, r and the weights; each body reads r and writes F
    row = T * d * esz
    stored, partial, total, counts = 1, False, 0, []
    for l in range(1, L + 2):
        if l == 1:
            S = 1
            total += row + row
        else:
            total += stored * row + (row if partial else 0) + row   # reads
            total += row + row                                      # folded row, r
            closes = (l - 1) % B == 0 or l - 1 == L                 # v_{l-1} ends its block
            if closes:
                stored, partial = stored + 1, False
                S = stored
            else:
                partial = True
                S = stored + 1
        counts.append(S)
        total += T * S * 4
        if l <= L:
            total += 2 * row + 2 * d * 4
    return total, counts


def test_stack_byte_model_follows_the_state():
    from depth_wise_attention_block_gb300 import attnres_num_sources
    from depth_wise_attention_block_gb300.stack import stack_forward_bytes
    for T, d, esz, L, B in [(2048, 7168, 2, 93, 12), (2048, 7168, 2, 93, 1), (64, 7168, 2, 93, 12),
                            (8, 256, 4, 14, 4), (5, 64, 4, 7, 3), (3, 16, 2, 1, 1), (16, 32, 4, 30, 7)]:
        total, counts = _simulated_stack_bytes(T, d, esz, L, B)
        assert counts == [attnres_num_sources(l, B, L) for l in range(1, L + 2)]
        assert stack_forward_bytes(T, d, esz, L, B) == total
    # the figures the bench divides by: the K3 prefill stack and the Full
    # AttnRes stack (block size 1) at T = 2048
    assert stack_forward_bytes(2048, 7168, 2, 93, 12) == 28_195_168_256
    assert stack_forward_bytes(2048, 7168, 2, 93, 1) == 142_086_209_536
