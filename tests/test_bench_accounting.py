"""The benchmark's algorithmic byte counts (the numerators of every GB/s it
reports) against the sizes of oracle-packed arrays: what a decode launch must
read and write, with row padding excluded."""
import numpy as np
import pytest

import bench
import oracle


@pytest.mark.parametrize("N,K,G", [(16, 4096, 128), (24, 640, 128), (8, 768, 32), (40, 1536, 64), (8, 5120, 256)])
@pytest.mark.parametrize("M", [1, 3])
def test_gemv_bytes_are_codes_scales_zeros_x_y(M, N, K, G):
    q, s, z = oracle.pack(np.zeros((N, K), np.float16), G)
    ng = K // G
    unpadded_meta = N * ng * 2 + N * ng // 2          # one FP16 scale and one 4-bit zero per group
    assert q.nbytes == N * K // 2
    assert s.nbytes >= N * ng * 2 and z.nbytes * 2 >= N * ng   # the stored rows may be padded
    assert bench.gemv_bytes(M, N, K, G) == q.nbytes + unpadded_meta + M * K * 2 + M * N * 2


@pytest.mark.parametrize("N,K", [(8, 256), (24, 768), (16, 8192)])
@pytest.mark.parametrize("M", [1, 3])
def test_q4k_bytes_are_codes_records_x_y(M, N, K):
    q, meta = oracle.q4k_pack(np.zeros((N, K), np.float16))
    assert bench.q4k_bytes(M, N, K) == q.nbytes + meta.nbytes + M * K * 2 + M * N * 2
    assert (q.nbytes + meta.nbytes) * 8 / (N * K) == 4.5


def test_w8_bytes_count_both_planes_and_x_once():
    """The 8-bit layer's sweep rows count what the kernels read: the 2K-channel 4-bit layer of both planes
    (codes, both planes' scales and zeros) with x counted once."""
    M, N, K, G = 2, 16, 1024, 128
    q, s, z = oracle.pack8(np.zeros((N, K), np.float16), G)
    assert q.nbytes == N * K                                      # 8 bits per weight of codes
    counted = bench.gemv_bytes(M, N, 2 * K, G) - M * K * 2
    assert counted == q.nbytes + N * (2 * K // G) * 2 + N * (2 * K // G) // 2 + M * K * 2 + M * N * 2
