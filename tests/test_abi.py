"""The C ABI library loads, exports every symbol ``include/ringattn.h``
declares, and rejects bad arguments on the host before touching a GPU.
CPU only: no call here reaches a CUDA API."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


@pytest.fixture(scope="module")
def L():
    from ring_attention_fwd_gb300 import binding, build
    if not (os.path.exists(binding._LIB_PATH) and os.path.exists(binding._CHECKED_PATH)):
        build.build()
    return binding.lib()


@pytest.fixture(scope="module")
def LC(L):
    """The bounds-checked build (loaded beside the default one)."""
    from ring_attention_fwd_gb300 import binding
    return binding._load(binding._CHECKED_PATH)


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"RA_API\s+[\w\s\*]+?\b(ra_\w+)\s*\(", text)))


def test_header_declares_the_api():
    assert declared_symbols() == sorted([
        "ra_fwd", "ra_fwd_step", "ra_fwd_step_fold", "ra_merge", "ra_bwd_workspace_bytes", "ra_bwd", "ra_bwd_step", "ra_bwd_noalloc",
        "ra_decode_workspace_bytes", "ra_decode", "ra_ffn_workspace_bytes", "ra_ffn", "ra_set_timing_buffer",
        "ra_set_kernel_timing", "ra_kernel_times", "ra_set_wait_test", "ra_set_fwd_kernel", "ra_check_device_status",
        "ra_read_checks", "ra_last_error", "ra_version"])


def test_library_exports_every_declared_symbol(L):
    from ring_attention_fwd_gb300 import binding
    for name in declared_symbols():
        assert hasattr(L, name), name
        assert name in binding.SIGNATURES, name


def test_checked_build_exports_every_declared_symbol(LC):
    for name in declared_symbols():
        assert hasattr(LC, name), name
    assert LC.ra_version().decode().endswith("checked")


def test_version(L):
    assert L.ra_version().decode().startswith("ringattn")
    assert not L.ra_version().decode().endswith("checked")


def test_read_checks_only_in_checked_build(L, LC):
    from ring_attention_fwd_gb300 import binding
    rep = binding.CheckReport()
    assert L.ra_read_checks(ctypes.addressof(rep), None) == 2
    assert "not the checked build" in L.ra_last_error().decode()
    assert LC.ra_read_checks(None, None) == 1 and "null" in LC.ra_last_error().decode()
    assert ctypes.sizeof(binding.CheckReport) == 88


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(L, **kw):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, B=1, H=1, S=256, D=128, N=2, causal=1, layout=0, dtype=1, O=FAKE,
             LSE=FAKE, stream=None)
    a.update(kw)
    return L.ra_fwd(a["Q"], a["K"], a["V"], a["B"], a["H"], a["S"], a["D"], a["N"], a["causal"], a["layout"],
                    a["dtype"], a["O"], a["LSE"], a["stream"])


@pytest.mark.parametrize("kw,code,needle", [
    (dict(Q=None), 1, "null"),
    (dict(LSE=None), 1, "null"),
    (dict(S=255), 1, "multiple of N"),
    (dict(N=0), 1, ">= 1"),
    (dict(B=0), 1, ">= 1"),
    (dict(causal=2), 1, "causal"),
    (dict(layout=7), 1, "layout"),
    (dict(dtype=9), 1, "dtype"),
    (dict(D=64), 2, "D == 128"),
    (dict(dtype=0, D=130), 2, "D % 4"),
    (dict(Q=FAKE + 8), 1, "16-byte"),
    (dict(LSE=FAKE + 2), 1, "4-byte"),
    (dict(B=2**31, H=2), 1, "2^31"),
    (dict(S=2**40, N=1, H=2**20), 1, "2^31-1"),
])
def test_fwd_rejects_bad_arguments(L, kw, code, needle):
    assert _fwd(L, **kw) == code
    assert needle in L.ra_last_error().decode()


def test_merge_rejects_bad_arguments(L):
    assert L.ra_merge(FAKE, FAKE, FAKE, FAKE, 0, 128, 1, None) == 0       # rows == 0: no-op
    assert L.ra_merge(FAKE, FAKE, FAKE, FAKE, -1, 128, 1, None) == 1
    assert L.ra_merge(FAKE, FAKE, FAKE, FAKE, 4, 0, 1, None) == 1
    assert L.ra_merge(FAKE, FAKE, FAKE, FAKE, 4, 2048, 1, None) == 1
    assert L.ra_merge(None, FAKE, FAKE, FAKE, 4, 128, 1, None) == 1
    assert L.ra_merge(FAKE, FAKE + 2, FAKE, FAKE, 4, 128, 1, None) == 1
    assert L.ra_merge(FAKE, FAKE, FAKE, FAKE, 4, 128, 5, None) == 1


def test_bwd_workspace_size(L):
    up = lambda x: (x + 255) // 256 * 256
    B, H, S, D, N = 1, 32, 65536, 128, 16
    padded = N * ((S // N + 127) // 128) * 128
    assert L.ra_bwd_workspace_bytes(B, H, S, D, N) == 2 * up(B * H * padded * 4)
    # ragged blocks: 3 blocks of 200 rows -> 2 query tiles of 128 each per block
    assert L.ra_bwd_workspace_bytes(1, 2, 600, 128, 3) == 2 * up(2 * 3 * 256 * 4)
    assert L.ra_bwd_workspace_bytes(0, 1, 1, 1, 1) == 0
    assert L.ra_bwd_workspace_bytes(1, 1, 10, 128, 3) == 0      # S % N != 0


def test_bwd_rejects_bad_arguments(L):
    def call(**kw):
        a = dict(B=1, H=1, S=256, D=128, N=2, causal=1, layout=1, dtype=1, ws=FAKE, ws_bytes=1 << 30)
        a.update(kw)
        return L.ra_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["S"], a["D"],
                        a["N"], a["causal"], a["layout"], a["dtype"], a["ws"], a["ws_bytes"], None)
    assert call(ws=None) == 1
    assert call(S=100, N=3) == 1
    assert call(dtype=0) == 2
    assert call(D=64) == 2
    assert call(ws_bytes=16) == 1 and "workspace" in L.ra_last_error().decode()
    assert call(ws=FAKE + 16) == 1 and "256-byte" in L.ra_last_error().decode()


def test_bwd_noalloc_rejects_sizes_before_touching_a_gpu(L):
    def call(B, H, S, N):
        return L.ra_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, S, 128, N, 1, 0, 1,
                                None)
    assert call(1, 1, 100, 3) == 1 and "invalid sizes" in L.ra_last_error().decode()
    assert call(1, 64, 131072, 32) == 1 and "more than the fixed" in L.ra_last_error().decode()


def test_fwd_step_rejects_bad_block_indices(L):
    def call(N, i, j):
        return L.ra_fwd_step(FAKE, FAKE, FAKE, 1, 1, 64, 128, N, i, j, 1, 0, 1, FAKE, FAKE, None)
    assert call(4, 4, 0) == 1 and "0 <= i, j < N" in L.ra_last_error().decode()
    assert call(4, 0, -1) == 1
    assert call(0, 0, 0) == 1
    assert L.ra_fwd_step(None, FAKE, FAKE, 1, 1, 64, 128, 4, 1, 0, 1, 0, 1, FAKE, FAKE, None) == 1


def test_decode_workspace_size(L):
    """Per-chunk partials: D floats + 1 LSE per work item, each part rounded
    up to 256 bytes.  The split depends on the sizes only."""
    up = lambda x: (x + 255) // 256 * 256

    def expect(B, H, S, D, N):
        bh, c = B * H, -(-S // N)
        want = max(1, -(-(16 * 152) // (bh * N)))
        chunk = max(-(-(-(-c // want)) // 64) * 64, min(-(-c // 64) * 64, 256))
        items = bh * N * -(-c // chunk)
        return up(items * D * 4) + up(items * 4)

    for args in [(1, 32, 262144, 128, 32), (2, 3, 1000, 128, 3), (1, 1, 1, 128, 1), (1, 2, 5, 128, 9),
                 (4, 8, 65536, 128, 1)]:
        assert L.ra_decode_workspace_bytes(*args) == expect(*args), args
    assert L.ra_decode_workspace_bytes(1, 32, 262144, 128, 32) == up(3072 * 128 * 4) + up(3072 * 4)
    assert L.ra_decode_workspace_bytes(0, 1, 1, 128, 1) == 0
    assert L.ra_decode_workspace_bytes(1, 1, 0, 128, 1) == 0


def test_decode_rejects_bad_arguments(L):
    def call(**kw):
        a = dict(q=FAKE, B=1, H=2, S=300, D=128, N=4, dtype=1, O=FAKE, LSE=FAKE, ws=FAKE, ws_bytes=1 << 30)
        a.update(kw)
        return L.ra_decode(a["q"], FAKE, FAKE, a["B"], a["H"], a["S"], a["D"], a["N"], a["dtype"], a["O"],
                           a["LSE"], a["ws"], a["ws_bytes"], None)
    assert call(q=None) == 1 and "null" in L.ra_last_error().decode()
    assert call(S=0) == 1 and "invalid sizes" in L.ra_last_error().decode()
    assert call(N=0) == 1
    assert call(dtype=7) == 1
    assert call(dtype=0) == 2
    assert call(D=64) == 2
    assert call(q=FAKE + 8) == 1 and "16-byte" in L.ra_last_error().decode()
    assert call(LSE=FAKE + 2) == 1
    assert call(ws=FAKE + 16) == 1 and "256-byte" in L.ra_last_error().decode()
    assert call(ws_bytes=16) == 1 and "workspace" in L.ra_last_error().decode()


def test_bwd_step_rejects_bad_arguments(L):
    def call(N=4, i=1, j=0, causal=1, layout=0, dtype=1, D=128, ws=FAKE, ws_bytes=1 << 30, c=256):
        return L.ra_bwd_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, c, D, N, i, j, causal,
                             layout, dtype, ws, ws_bytes, None)
    assert call(i=4) == 1 and "0 <= i, j < N" in L.ra_last_error().decode()
    assert call(j=-1) == 1
    assert call(N=0) == 1
    assert call(layout=5) == 1
    assert call(dtype=0) == 2
    assert call(D=64) == 2
    assert call(ws_bytes=16) == 1 and "workspace" in L.ra_last_error().decode()
    assert call(c=0) == 1
    # contiguous causal j > i: nothing to add, returns before touching memory
    assert call(i=0, j=3) == 0
    assert L.ra_bwd_step(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 128, 4, 0, 3, 1, 0, 1,
                         FAKE, 1 << 30, None) == 1


def test_ffn_workspace_and_bad_arguments(L):
    up = lambda x: (x + 255) // 256 * 256
    assert L.ra_ffn_workspace_bytes(16384, 4096, 11008, 4096) == 4096 * 11008 * 2 + 256   # + 8 tile counters
    assert L.ra_ffn_workspace_bytes(100, 256, 128, 4096) == up(100 * 128 * 2) + 256
    assert L.ra_ffn_workspace_bytes(100000, 256, 128, 1000) == up(1000 * 128 * 2) + up(2 * 100 * 4)
    assert L.ra_ffn_workspace_bytes(100, 255, 128, 64) == 0
    assert L.ra_ffn_workspace_bytes(100, 256, 100, 64) == 0

    def call(T=300, h=256, f=384, c=128, dtype=1, ws=FAKE, ws_bytes=1 << 30, X=FAKE):
        return L.ra_ffn(X, FAKE, FAKE, FAKE, FAKE, T, h, f, c, dtype, ws, ws_bytes, None)
    assert call(X=None) == 1 and "null" in L.ra_last_error().decode()
    assert call(h=384) == 1 and "multiple of 256" in L.ra_last_error().decode()
    assert call(f=200) == 1
    assert call(T=0) == 1
    assert call(c=0) == 1
    assert call(dtype=0) == 2
    assert call(dtype=5) == 1
    assert call(X=FAKE + 8) == 1 and "16-byte" in L.ra_last_error().decode()
    assert call(ws=FAKE + 16) == 1 and "256-byte" in L.ra_last_error().decode()
    assert call(ws_bytes=1000) == 1 and "workspace" in L.ra_last_error().decode()


def test_wait_test_switch_arguments(L):
    assert L.ra_set_wait_test(3) == 1
    assert L.ra_set_wait_test(0) == 0


def test_fwd_kernel_switch_arguments(L):
    from ring_attention_fwd_gb300 import binding
    assert L.ra_set_fwd_kernel(2) == 1 and "RA_FWD_PAIR" in L.ra_last_error().decode()
    assert L.ra_set_fwd_kernel(-1) == 1
    for kind in (1, 0):                    # ends on the default
        assert L.ra_set_fwd_kernel(kind) == 0
    with pytest.raises(ValueError):
        binding.set_fwd_kernel("dual")


def test_kernel_timing_arguments(L):
    n = ctypes.c_int(-1)
    assert L.ra_set_kernel_timing(2) == 1
    assert L.ra_kernel_times(None, -1, ctypes.byref(n)) == 1
    assert L.ra_kernel_times(None, 0, ctypes.byref(n)) == 0 and n.value == 0   # nothing recorded
    assert L.ra_set_kernel_timing(0) == 0


def test_timing_buffer_arguments(L):
    assert L.ra_set_timing_buffer(FAKE, 0) == 1
    assert L.ra_set_timing_buffer(None, 0) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from ring_attention_fwd_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no non-CUDA fallback"):
        binding.lib()


def test_fwd_step_fold_rejects_bad_arguments(L):
    def call(**kw):
        a = dict(Q=FAKE, K=FAKE, V=FAKE, B=1, H=1, c=128, D=128, N=4, i=1, j=0, causal=1, layout=0, dtype=1,
                 O=FAKE, L=FAKE)
        a.update(kw)
        return L.ra_fwd_step_fold(a["Q"], a["K"], a["V"], a["B"], a["H"], a["c"], a["D"], a["N"], a["i"], a["j"],
                                  a["causal"], a["layout"], a["dtype"], a["O"], a["L"], None)
    assert call(O=None) == 1 and "null" in L.ra_last_error().decode()
    assert call(L=None) == 1
    assert call(i=4) == 1 and "0 <= i, j < N" in L.ra_last_error().decode()
    assert call(j=-1) == 1
    assert call(dtype=0, i=0, j=3) == 2          # contiguous causal j > i: sizes and dtype still checked
    assert call(i=0, j=3) == 0                   # ... and then nothing to fold, no launch
    assert call(O=FAKE + 4) == 1 and "16-byte" in L.ra_last_error().decode()
