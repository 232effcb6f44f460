"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/w4a16.h declares, and rejects bad arguments on the host before
touching any device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import w4a16_weight_only_linear_b300 as w4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"W4A16_API\s+[\w\s\*]+?\b((?:w[48]a16|q4k)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("w4a16_pack", "w4a16_linear", "w4a16_linear_dual", "w4a16_dequant", "w4a16_status_string"):
        assert required in names
    assert set(names) == set(w4.EXPORTS), "binding and header disagree"


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(w4.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else():
    # the build hides everything but the declared C entry points
    out = os.popen(f"nm -D --defined-only {w4.LIB_PATH}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith(("w4a16", "w8a16", "q4k"))}
    assert ours == set(declared_symbols())


def test_status_strings():
    assert w4.w4a16_status_string(0) == "W4A16_OK"
    for code, name in w4.STATUS_NAMES.items():
        assert w4.w4a16_status_string(code) == name
    assert w4.w4a16_status_string(99) == "W4A16_ERR_UNKNOWN"


@pytest.mark.parametrize("K,G", [(4096, 128), (5120, 128), (13824, 128), (5120, 32), (5120, 64), (5120, 256),
                                 (64, 32), (96, 32)])
def test_layout_helpers(K, G):
    ng = K // G
    assert w4.w4a16_qweight_ld(K) == K // 8
    lds = w4.w4a16_scales_ld(K, G)
    ldz = w4.w4a16_zeros_ld(K, G)
    assert lds >= ng and lds % 8 == 0 and lds - ng < 8            # 16-byte rows of halves
    assert ldz >= (ng + 7) // 8 and ldz % 4 == 0 and ldz - (ng + 7) // 8 < 4


def _call_linear(fn, x=1 << 12, q=1 << 12, s=1 << 12, z=1 << 12, M=1, N=64, K=256, G=128, y=1 << 12):
    # fake, never-dereferenced addresses: every call here must fail validation
    v = ctypes.c_void_p
    return getattr(w4._lib, fn)(v(x), v(q), v(s), v(z), M, N, K, G, v(y), v(0))


@pytest.mark.parametrize("fn", ["w4a16_linear", "w4a16_linear_gemv", "w4a16_linear_gemm"])
def test_linear_argument_errors(fn):
    assert _call_linear(fn, G=48) == 2                  # unsupported group size
    assert _call_linear(fn, G=512) == 2
    assert _call_linear(fn, K=200) == 1                 # K % G
    assert _call_linear(fn, N=60) == 1                  # N % 8
    assert _call_linear(fn, K=0) == 1
    assert _call_linear(fn, M=-1) == 1
    assert _call_linear(fn, x=0) == 1                   # null pointers
    assert _call_linear(fn, q=0) == 1
    assert _call_linear(fn, y=0) == 1
    assert _call_linear(fn, x=(1 << 12) + 8) == 3      # misaligned
    assert _call_linear(fn, s=(1 << 12) + 2) == 3
    assert _call_linear(fn, M=0) == 0                   # empty problem: nothing launched
    assert _call_linear(fn, N=0) == 0


def test_dequant_debug_is_the_dequant_call():
    # same validation as w4a16_dequant (no compute call here): bad group, N % 8, misaligned output, empty
    v = ctypes.c_void_p
    a = v(1 << 12)
    for name in ("w4a16_dequant", "w4a16_dequant_debug"):
        f = getattr(w4._lib, name)
        assert f(a, a, a, 64, 256, 100, a, v(0)) == 2
        assert f(a, a, a, 60, 256, 128, a, v(0)) == 1
        assert f(a, a, a, 64, 256, 128, v((1 << 12) + 4), v(0)) == 3
        assert f(a, a, a, 0, 256, 128, a, v(0)) == 0


def test_pack_and_dequant_argument_errors():
    v = ctypes.c_void_p
    a = v(1 << 12)
    assert w4._lib.w4a16_pack(a, 64, 256, 100, a, a, a, v(0)) == 2
    assert w4._lib.w4a16_pack(a, 60, 256, 128, a, a, a, v(0)) == 1
    assert w4._lib.w4a16_pack(v(0), 64, 256, 128, a, a, a, v(0)) == 1
    assert w4._lib.w4a16_pack(v((1 << 12) + 4), 64, 256, 128, a, a, a, v(0)) == 3
    assert w4._lib.w4a16_pack(a, 0, 256, 128, a, a, a, v(0)) == 0
    assert w4._lib.w4a16_dequant(a, a, a, 64, 250, 128, a, v(0)) == 1
    assert w4._lib.w4a16_dequant(a, a, a, 64, 256, 128, v(0), v(0)) == 1


def test_dequant_f16_and_q4k_dequant_argument_errors():
    v = ctypes.c_void_p
    a = v(1 << 12)
    f = w4._lib.w4a16_dequant_f16
    assert f(a, a, a, 64, 256, 100, a, v(0)) == 2
    assert f(a, a, a, 60, 256, 128, a, v(0)) == 1
    assert f(a, a, a, 64, 256, 128, v(0), v(0)) == 1
    assert f(a, a, a, 64, 256, 128, v((1 << 12) + 4), v(0)) == 3
    assert f(a, a, a, 0, 256, 128, a, v(0)) == 0
    g = w4._lib.q4k_dequant
    assert g(a, a, 64, 300, a, v(0)) == 1                # K % 256
    assert g(a, a, 60, 256, a, v(0)) == 1                # N % 8
    assert g(a, v(0), 64, 256, a, v(0)) == 1
    assert g(a, a, 64, 256, v((1 << 12) + 8), v(0)) == 3
    assert g(a, a, 0, 256, a, v(0)) == 0


def test_linear_f32_argument_errors():
    v = ctypes.c_void_p
    a = v(1 << 12)
    f = w4._lib.w4a16_linear_f32
    for path in (0, 1, 2):
        assert f(a, a, a, a, 1, 64, 256, 48, path, a, v(0)) == 2
        assert f(a, a, a, a, 1, 60, 256, 128, path, a, v(0)) == 1
        assert f(a, a, a, a, 1, 64, 256, 128, path, v(0), v(0)) == 1
        assert f(a, a, a, a, 1, 64, 256, 128, path, v((1 << 12) + 4), v(0)) == 3
        assert f(a, a, a, a, 0, 64, 256, 128, path, a, v(0)) == 0
    assert f(a, a, a, a, 1, 64, 256, 128, 3, a, v(0)) == 1          # no such path
    assert f(a, a, a, a, 1, 64, 256, 128, -1, a, v(0)) == 1


def test_dual_argument_errors():
    v = ctypes.c_void_p
    a = v(1 << 12)
    f = w4._lib.w4a16_linear_dual
    assert f(a, a, a, a, a, a, a, 1, 64, 256, 96, a, a, v(0)) == 2
    assert f(a, a, a, a, v(0), a, a, 1, 64, 256, 128, a, a, v(0)) == 1
    assert f(a, a, a, a, a, a, a, 1, 64, 256, 128, a, v((1 << 12) + 2), v(0)) == 3
    assert f(a, a, a, a, a, a, a, 0, 64, 256, 128, a, a, v(0)) == 0


def test_w8a16_word_layout_and_argument_errors():
    for K, G in ((4096, 128), (5120, 32), (13824, 128), (64, 32), (96, 32), (768, 256)):
        ng = K // G
        assert w4._lib.w8a16_qweight_ld(K) == K // 4
        assert w4._lib.w8a16_scales_ld(K, G) == w4.w4a16_scales_ld(K, G)
        ldz = w4._lib.w8a16_zeros_ld(K, G)
        assert ldz >= (ng + 3) // 4 and ldz % 4 == 0 and ldz - (ng + 3) // 4 < 4        # 16-byte rows
    v = ctypes.c_void_p
    a = v(1 << 12)
    assert w4._lib.w8a16_pack(a, 64, 256, 100, a, a, a, v(0)) == 2
    assert w4._lib.w8a16_pack(a, 60, 256, 128, a, a, a, v(0)) == 1
    assert w4._lib.w8a16_pack(v((1 << 12) + 4), 64, 256, 128, a, a, a, v(0)) == 3
    assert w4._lib.w8a16_pack(a, 0, 256, 128, a, a, a, v(0)) == 0
    for fn in ("w8a16_linear", "w8a16_linear_gemv", "w8a16_linear_gemm"):
        assert _call_linear(fn, G=48) == 2
        assert _call_linear(fn, K=200) == 1
        assert _call_linear(fn, x=0) == 1
        assert _call_linear(fn, s=(1 << 12) + 2) == 3
        assert _call_linear(fn, M=0) == 0
    for fn in ("w8a16_dequant", "w8a16_dequant_f16"):
        f = getattr(w4._lib, fn)
        assert f(a, a, a, 64, 256, 100, a, v(0)) == 2
        assert f(a, a, a, 60, 256, 128, a, v(0)) == 1
        assert f(a, a, a, 64, 256, 128, v((1 << 12) + 4), v(0)) == 3
        assert f(a, a, a, 0, 256, 128, a, v(0)) == 0


def test_w8a16_planes_layout_and_argument_errors():
    for K, G in ((4096, 128), (5120, 32), (13824, 128), (64, 32)):
        assert w4._lib.w8a16_planes_qweight_ld(K) == K // 4
        assert w4._lib.w8a16_planes_scales_ld(K, G) == w4.w4a16_scales_ld(2 * K, G)
        assert w4._lib.w8a16_planes_zeros_ld(K, G) == w4.w4a16_zeros_ld(2 * K, G)
    v = ctypes.c_void_p
    a = v(1 << 12)
    assert w4._lib.w8a16_planes_pack(a, 64, 256, 100, a, a, a, v(0)) == 2
    assert w4._lib.w8a16_planes_pack(a, 60, 256, 128, a, a, a, v(0)) == 1
    assert w4._lib.w8a16_planes_pack(v((1 << 12) + 4), 64, 256, 128, a, a, a, v(0)) == 3
    assert w4._lib.w8a16_planes_pack(a, 0, 256, 128, a, a, a, v(0)) == 0
    assert _call_linear("w8a16_planes_linear", G=48) == 2
    assert _call_linear("w8a16_planes_linear", K=200) == 1
    assert _call_linear("w8a16_planes_linear", x=0) == 1
    assert _call_linear("w8a16_planes_linear", s=(1 << 12) + 2) == 3
    assert _call_linear("w8a16_planes_linear", M=0) == 0


def test_q4k_layout_and_argument_errors():
    for K in (256, 4096, 8192, 28672):
        assert w4._lib.q4k_meta_ld(K) == K // 256 * 4
    assert w4._lib.q4k_meta_ld(384) == 0 and w4._lib.q4k_meta_ld(0) == 0
    assert w4.q4k_packed_shapes(64, 512) == ((64, 64), (64, 8))
    v = ctypes.c_void_p
    a = v(1 << 12)
    p = w4._lib.q4k_pack
    assert p(a, 64, 384, a, a, v(0)) == 1                      # K % 256
    assert p(a, 60, 256, a, a, v(0)) == 1                      # N % 8
    assert p(a, 64, 256, a, v(0), v(0)) == 1                   # null meta
    assert p(v((1 << 12) + 2), 64, 256, a, a, v(0)) == 3       # misaligned w
    assert p(a, 64, 256, a, v((1 << 12) + 4), v(0)) == 3       # misaligned meta
    assert p(a, 0, 256, a, a, v(0)) == 0                       # empty
    f = w4._lib.q4k_linear
    assert f(a, a, a, 1, 64, 384, a, v(0)) == 1
    assert f(a, a, a, 1, 60, 256, a, v(0)) == 1
    assert f(a, a, a, -1, 64, 256, a, v(0)) == 1
    assert f(v(0), a, a, 1, 64, 256, a, v(0)) == 1
    assert f(a, v((1 << 12) + 8), a, 1, 64, 256, a, v(0)) == 3
    assert f(a, a, a, 1, 64, 256, v((1 << 12) + 2), v(0)) == 3
    assert f(a, a, a, 0, 64, 256, a, v(0)) == 0
    d = w4._lib.q4k_linear_dual
    assert d(a, a, a, a, v(0), 1, 64, 256, a, a, v(0)) == 1
    assert d(a, a, a, a, a, 1, 64, 512 + 128, a, a, v(0)) == 1
    assert d(a, a, a, a, a, 1, 64, 256, a, v((1 << 12) + 2), v(0)) == 3
    assert d(a, a, a, a, a, 0, 64, 256, a, a, v(0)) == 0


def test_act_scaled_argument_errors():
    v = ctypes.c_void_p
    a = v(1 << 12)
    f = w4._lib.w4a16_linear_act_scaled
    assert f(a, a, a, a, a, 1, 64, 256, 96, a, v(0)) == 2                  # unsupported group size
    assert f(a, v(0), a, a, a, 1, 64, 256, 128, a, v(0)) == 1              # null x_scale
    assert f(a, v((1 << 12) + 4), a, a, a, 1, 64, 256, 128, a, v(0)) == 3  # misaligned x_scale
    assert f(a, a, a, a, a, 1, 60, 256, 128, a, v(0)) == 1                 # N % 8
    assert f(v(0), a, a, a, a, 1, 64, 256, 128, a, v(0)) == 1              # null x
    assert f(a, a, a, a, a, 0, 64, 256, 128, a, v(0)) == 0                 # empty problem
    d = w4._lib.w4a16_linear_dual_act_scaled
    assert d(a, v(0), a, a, a, a, a, a, 1, 64, 256, 128, a, a, v(0)) == 1
    assert d(a, v((1 << 12) + 8), a, a, a, a, a, a, 1, 64, 256, 128, a, a, v(0)) == 3
    assert d(a, a, a, a, a, a, a, a, 1, 64, 256, 96, a, a, v(0)) == 2
    assert d(a, a, a, a, a, a, a, a, 0, 64, 256, 128, a, a, v(0)) == 0


def test_path_query_rejects_bad_shapes():
    assert w4.w4a16_linear_path(1, 60, 256, 128) == 0
    assert w4.w4a16_linear_path(1, 64, 250, 128) == 0
    assert w4.w4a16_linear_path(1, 64, 256, 100) == 0


@pytest.mark.parametrize("N,K", [(4096, 4096), (5120, 5120), (13824, 5120), (5120, 13824), (28672, 8192),
                                 (8192, 28672)])
@pytest.mark.parametrize("G", [32, 64, 128, 256])
def test_dispatch_rule(N, K, G):
    """Host-only dispatch: the decode GEMV up to M = 8 where its x staging and tables fit, and up to
    M = 16 where it runs with all its warps; the tensor-core GEMM above.  M = 1 fits at every workload
    shape, and once a batch size leaves the GEMV every larger one does too."""
    paths = [w4.w4a16_linear_path(M, N, K, G) for M in range(1, 20)]
    assert set(paths) <= {1, 2}
    assert paths[0] == 1
    assert all(p == 2 for p in paths[16:])                     # M >= 17
    first_gemm = paths.index(2)
    assert all(p == 2 for p in paths[first_gemm:])
    assert w4.w4a16_linear_path(2048, N, K, G) == 2


def test_gemv_plan_query():
    """The planner's choices on a B300 (148 SMs, 227 KB of shared memory; on a GPU the device's own
    figures): the 70B decode geometry, the K split where x would crowd out the rings, and errors."""
    plan = (ctypes.c_int32 * 6)()

    def q(M, N, K, G, mode=0):
        st = w4._lib.w4a16_debug_gemv_plan(M, N, K, G, mode, plan)
        return st, list(plan)

    st, p = q(1, 28672, 8192, 128)
    assert st == 0 and p[:4] == [4, 2, 16, 0] and p[4] == 148
    st, p = q(16, 13824, 5120, 128)                     # x = 160 KB: split over clusters of two
    assert st == 0 and p[0] == 1 and p[3] == 1 and p[4] % 2 == 0 and p[2] == 12
    st, p = q(12, 13824, 5120, 128)                     # x = 120 KB: the plain kernel keeps all its warps
    assert st == 0 and p[3] == 0 and p[2] == 12
    st, p = q(8, 264, 13824, 128)                       # x = 221 KB: only the split fits
    assert st == 0 and p[:2] == [1, 1] and p[3] == 1
    assert q(16, 28672, 8192, 128)[0] == 2              # unsupported: even half of x leaves no room
    assert q(17, 264, 1024, 128)[0] == 1                # M outside 1..16
    assert q(1, 60, 1024, 128)[0] == 1                  # N not a multiple of 8
    assert q(16, 13824, 5120, 128, 1)[1][2] == 4       # the plain kernel there: 4 warps
    assert q(8, 264, 13824, 128, 1)[0] == 2             # ... and no plain plan at all
    assert q(1, 264, 1024, 128, 3)[0] == 1              # mode outside 0..2
    assert w4._lib.w4a16_debug_gemv_plan(1, 264, 1024, 128, 0, None) == 1


def test_dispatch_falls_back_when_the_gemv_does_not_fit():
    # x is staged as M*K FP16 beside the resident metadata rows: at K = 65536 one row still fits at
    # G = 32 (whose scales stream with the weights; only the zero rows stay resident) and G = 128,
    # not at G = 64 (resident scales and zeros); at K = 98304 the staged x alone leaves no room
    assert w4.w4a16_linear_path(1, 8192, 65536, 32) == 1
    assert w4.w4a16_linear_path(1, 8192, 65536, 64) == 2
    assert w4.w4a16_linear_path(1, 8192, 65536, 128) == 1
    for G in (32, 64, 128, 256):
        assert w4.w4a16_linear_path(1, 8192, 98304, G) == 2


def test_withhold_hook_rejects_unknown_kernels():
    assert w4._lib.w4a16_debug_withhold_copy(3) == 1
    assert w4._lib.w4a16_debug_withhold_copy(-1) == 1
    assert w4._lib.w4a16_debug_withhold_copy(0) == 0          # disarmed
    w4._lib.w4a16_debug_set_wait_limit(0)                      # default budget


def test_entry_points_from_several_threads():
    """The host-side state (device attributes, tensor-map cache, per-kernel
    attribute caches, the test hooks) is shared by every thread; calls from
    several threads at once must give each caller its own, correct answer.
    Without a GPU only the host paths run: dispatch queries, layout helpers and
    argument validation."""
    import threading
    v = ctypes.c_void_p
    a = v(1 << 12)
    expect = {(M, N, K, G): w4.w4a16_linear_path(M, N, K, G)
              for M in (1, 4, 8, 16, 300) for N in (264, 4096, 13824) for K in (1024, 5120) for G in (32, 128)}
    errors = []

    def worker(seed):
        try:
            for i in range(300):
                for key, path in expect.items():
                    if w4.w4a16_linear_path(*key) != path:
                        errors.append(("path", key))
                K = 256 * (1 + (i + seed) % 8)
                if w4.w4a16_scales_ld(K, 128) != ((K // 128 + 7) // 8) * 8:
                    errors.append(("lds", K))
                if w4._lib.w4a16_linear(a, a, a, a, 1, 60, K, 128, a, v(0)) != 1:
                    errors.append(("validate", K))
        except Exception as e:          # pragma: no cover - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:5]


def test_multi_argument_errors():
    v = ctypes.c_void_p
    a = 1 << 12
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    ns = lambda *n: (ctypes.c_int64 * len(n))(*n)
    f = w4._lib.w4a16_linear_multi
    q3, s3, z3, y3 = arr(a, a, a), arr(a, a, a), arr(a, a, a), arr(a, a, a)
    assert f(v(a), 0, q3, s3, z3, ns(64, 64, 64), 1, 256, 128, y3, v(0)) == 1      # nmat outside 1..4
    assert f(v(a), 5, q3, s3, z3, ns(64, 64, 64), 1, 256, 128, y3, v(0)) == 1
    assert f(v(a), 3, None, s3, z3, ns(64, 64, 64), 1, 256, 128, y3, v(0)) == 1    # null array
    assert f(v(a), 3, q3, s3, z3, None, 1, 256, 128, y3, v(0)) == 1
    assert f(v(a), 3, q3, s3, z3, ns(64, 60, 64), 1, 256, 128, y3, v(0)) == 1     # N % 8
    assert f(v(a), 3, q3, s3, z3, ns(64, 64, 64), 1, 256, 96, y3, v(0)) == 2       # group size
    assert f(v(a), 3, q3, s3, z3, ns(64, 64, 64), 1, 250, 128, y3, v(0)) == 1      # K % G
    assert f(v(a), 3, arr(a, 0, a), s3, z3, ns(64, 64, 64), 1, 256, 128, y3, v(0)) == 1
    assert f(v(a), 3, q3, s3, z3, ns(64, 64, 64), 1, 256, 128, arr(a, a + 2, a), v(0)) == 3
    assert f(v(a + 8), 3, q3, s3, z3, ns(64, 64, 64), 1, 256, 128, y3, v(0)) == 3
    assert f(v(a), 3, q3, s3, z3, ns(64, 64, 64), 0, 256, 128, y3, v(0)) == 0      # empty problem
    assert f(v(a), 3, q3, s3, z3, ns(0, 0, 0), 1, 256, 128, y3, v(0)) == 0


def test_host_planning_cost_of_a_call():
    """The host side of a call is planning, two cached tensor-map lookups and the launch.  The
    planning part runs here without a GPU (the path query plans both kernels for the shape): it
    must stay far below a decode launch's 25 us, or the host falls behind the GPU in a decode loop."""
    import time
    for _ in range(200):
        w4.w4a16_linear_path(1, 28672, 8192, 128)
    n = 5000
    t = time.perf_counter()
    for _ in range(n):
        w4.w4a16_linear_path(1, 28672, 8192, 128)
    us = (time.perf_counter() - t) / n * 1e6
    assert us < 20.0, f"{us:.1f} us per path query"
