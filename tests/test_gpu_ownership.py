"""What the library keeps between calls, and calls from several host threads.

  * The tensor-core path's FP16 copy of x comes from the device's current
    memory pool, stream-ordered, and is freed on the stream after the call:
    after the stream is synchronised the device's free memory is back where it
    was (the default pool releases at synchronisation), so the library holds no
    memory of its own between calls.
  * Several host threads calling the layer at once, each on its own stream,
    get the same outputs as calls made one at a time (the host caches of
    device attributes, tensor maps and kernel attributes are shared).
"""
import threading

import pytest
import torch

import oracle
import workloads as wl
from helpers import dev_packed

w4 = pytest.importorskip("w4a16_weight_only_linear_b300")

pytestmark = pytest.mark.gpu


def _problem(M, N, K, G, seed):
    w = wl.weight_f16(N, K, 0.02, seed)
    x = wl.activations_bf16(M, K, seed + 50)
    q, s, z = oracle.pack(wl.bits_u16(w), G)
    return x.cuda(), dev_packed(q, s, z)


def test_device_memory_returns_after_a_prefill_call():
    M, N, K, G = 2048, 1024, 8192, 128                  # x copy: 32 MiB
    x, dq = _problem(M, N, K, G, seed=31)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    w4.w4a16_linear(x, *dq, G, out=y)                   # loads the kernels' code
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        w4.w4a16_linear(x, *dq, G, out=y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"{(free0 - free1) / 2**20:.1f} MiB still held after the calls"
    assert w4.w4a16_device_status() == 0


def test_calls_from_several_threads_on_their_own_streams():
    cases = [(1, 1032, 4096, 128), (4, 520, 2048, 64), (300, 264, 1280, 128), (64, 1032, 4096, 32)]
    probs = [_problem(*c, seed=70 + i) for i, c in enumerate(cases)]
    want = []
    for (M, N, K, G), (x, dq) in zip(cases, probs):
        want.append(w4.w4a16_linear(x, *dq, G))
    torch.cuda.synchronize()
    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for r in range(20):
                    i = (t + r) % len(cases)
                    (M, N, K, G), (x, dq) = cases[i], probs[i]
                    y = w4.w4a16_linear(x, *dq, G, stream=stream)
                    stream.synchronize()
                    if not torch.equal(y, want[i]):
                        errors.append((t, r, cases[i]))
        except Exception as e:      # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors[:5]
    assert w4.w4a16_device_status() == 0


def test_host_time_per_decode_call_through_the_binding():
    """A decode call's host cost (binding, planning, cached tensor maps, launch), measured without
    synchronising: it must stay below the GPU time of the call it launches (about 25 us on the 70B
    shapes), or an eager decode loop becomes host-bound."""
    import time
    N, K, G = 28672, 8192, 128
    w = wl.weight_f16(N, K, 0.015, 5)
    q, s, z = w4.w4a16_pack(w.cuda(), G)
    x = wl.activations_bf16(1, K, 6).cuda()
    y = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(50):
        w4.w4a16_linear(x, q, s, z, G, out=y, stream=stream)
    torch.cuda.synchronize()
    n = 400
    t = time.perf_counter()
    for _ in range(n):
        w4.w4a16_linear(x, q, s, z, G, out=y, stream=stream)
    host_us = (time.perf_counter() - t) / n * 1e6
    torch.cuda.synchronize()
    assert host_us < 20.0, f"{host_us:.1f} us of host time per call"
    assert w4.w4a16_device_status() == 0
