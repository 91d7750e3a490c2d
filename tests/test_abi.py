"""The C-ABI library builds, loads and exports what include/pa_q8.h declares;
argument errors come back as status codes before any CUDA call (these run
on a machine without a GPU)."""
import ctypes
import shutil

import pytest

import int8_paged_kv_gb300 as pk
from int8_paged_kv_gb300 import _binding

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="needs nvcc to build the library")


@pytest.fixture(scope="module")
def L():
    from int8_paged_kv_gb300 import build
    build.build()
    return _binding.lib()


def test_exports_every_declared_function(L):
    names = _binding.header_functions()
    assert "pa_q8_decode" in names and "pa_q8_reshape_and_cache" in names
    for n in names:
        assert hasattr(L, n), f"libpa_q8.so does not export {n}"


def test_status_strings_and_version(L):
    assert pk.pa_q8_status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert pk.pa_q8_status_string(code) not in ("", "unknown status")
    assert pk.pa_q8_status_string(-99) == "unknown status"
    assert pk.pa_q8_version() >= 10000


ALIGNED = ctypes.c_void_p(0x10000)      # never dereferenced: every call below fails its checks first
MISALIGNED = ctypes.c_void_p(0x10004)


def _decode(L, *, out=ALIGNED, q=ALIGNED, kc=ALIGNED, S=2, H=8, Hk=2, D=128, B=16, Nb=4, nblocks=8):
    return L.pa_q8_decode(out, q, kc, ALIGNED, ALIGNED, ALIGNED, S, H, Hk, D, B, Nb, nblocks,
                          ctypes.c_float(0.1), None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(S=0), -1), (dict(H=0), -1), (dict(Hk=3), -1), (dict(D=66), -1), (dict(B=6), -1),
    (dict(Nb=0), -1), (dict(nblocks=0), -1), (dict(D=96), -2), (dict(B=12), -2), (dict(B=2048), -2),
    (dict(out=ctypes.c_void_p(0)), -1), (dict(q=MISALIGNED), -3), (dict(kc=MISALIGNED), -3),
])
def test_decode_argument_errors(L, kw, code):
    assert _decode(L, **kw) == code


def _writer(L, *, T=4, ks=512, vs=512, Hk=4, D=128, B=16, nb=8, key=ALIGNED, kc=ALIGNED):
    return L.pa_q8_reshape_and_cache(key, ALIGNED, kc, ALIGNED, ALIGNED, T, ks, vs, Hk, D, B, nb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), -1), (dict(Hk=0), -1), (dict(D=62), -1), (dict(B=2), -1), (dict(nb=0), -1),
    (dict(ks=100), -1), (dict(vs=511), -1), (dict(D=32, ks=128, vs=128), -2),
    (dict(key=ctypes.c_void_p(0)), -1), (dict(key=ctypes.c_void_p(0x10002)), -3),
    (dict(kc=ctypes.c_void_p(0x10001)), -3),
])
def test_writer_argument_errors(L, kw, code):
    assert _writer(L, **kw) == code


def test_writer_zero_tokens_is_a_noop(L):
    # no device work and no device query for an empty call
    assert _writer(L, T=0, key=ctypes.c_void_p(0)) == 0


def test_workspace_size_without_a_device(L):
    # size queries work without a GPU (they assume a 152-SM GB300)
    one = pk.pa_q8_decode_workspace_size(2, 4, 2, 64, 16, 7)                # one partition:
    assert 0 < one <= 256                                                    # just the sequence order
    long_ws = pk.pa_q8_decode_workspace_size(8, 32, 8, 128, 32, 4096)
    assert long_ws > 0 and long_ws % 4 == 0
    assert pk.pa_q8_decode_workspace_size(8, 32, 8, 100, 32, 4096) == 0     # invalid -> 0
    a = pk.pa_q8_decode_workspace_size(8, 32, 8, 128, 32, 4096, partition_tokens=1024)
    b = pk.pa_q8_decode_workspace_size(8, 32, 8, 128, 32, 4096, partition_tokens=4096)
    assert a > b > 0
    assert pk.pa_q8_decode_workspace_size(8, 32, 8, 128, 32, 4096, partition_tokens=100) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _binding.lib()


def test_contiguous_cache_shape_checks_without_a_device(L):
    import int8_paged_kv_gb300 as pk
    assert pk.pa_q8c_cache_words(100, 2, 128) == 100 * 256 // 4 + 100 * 256 // 32
    assert pk.pa_q8c_cache_words(100, 2, 100) == 0
    # head size 64: refused on the host (8-byte scale rows cannot be bulk-copied)
    rc = L.pa_q8c_decode(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 2, 8, 2, 64, 100, ctypes.c_float(0.1),
                         None, 0, None, None)
    assert rc == -2
    assert L.pa_q8c_decode(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 2, 8, 3, 128, 100, ctypes.c_float(0.1),
                           None, 0, None, None) == -1
    assert pk.pa_q8c_decode_workspace_size(4, 8, 2, 128, 4096) > 0
    assert pk.pa_q8c_decode_workspace_size(4, 8, 2, 64, 4096) == 0


def test_build_recompiles_when_its_flags_change(tmp_path):
    """The in-tree build records the compiler command it linked with; a later
    build with other flags (PA_Q8_NVCC_FLAGS) must treat every object as stale
    even though the objects are newer than their sources."""
    from int8_paged_kv_gb300 import build
    stamp = str(tmp_path / "flags.txt")
    key = "nvcc -gencode arch=compute_103a,code=sm_103a -O3"
    assert build._flags_changed(stamp, key)                       # never built here
    build._record_flags(stamp, key)
    assert not build._flags_changed(stamp, key)
    assert build._flags_changed(stamp, key + " -DPA_Q8_TC_WIDE=0")    # flags added
    build._record_flags(stamp, key + " -DX=1")
    assert build._flags_changed(stamp, key)                       # flags removed again
