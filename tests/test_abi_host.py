"""The C ABI without a GPU: libpi.so builds, loads, exports every entry point
include/pi.h declares, and rejects bad arguments on the host before any
launch (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import activation_sparse_decode_rank_gb300 as pi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pi.h")


@pytest.fixture(scope="module")
def lib():
    pi.build()
    return pi.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pi_[a-z_]+)\s*\(", src)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ["pi_predict", "pi_compact", "pi_sparse_ffn", "pi_dense_ffn", "pi_layer_decode",
              "pi_workspace_size", "pi_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libpi.so does not export {name}"
    # and the binding wraps each of them under the same name
    for name in declared_functions():
        assert name in pi.SIGNATURES
        assert callable(getattr(pi, name))


def test_status_strings(lib):
    for s in range(13):
        assert len(pi.status_string(s)) >= 2
    assert pi.status_string(0) == "ok"
    assert "unknown" in pi.status_string(99)


def test_workspace_size_host_only(lib):
    d = pi.make_desc(4096, 16384, 128, "f16")
    a = pi.pi_workspace_size(d, 1)
    b = pi.pi_workspace_size(d, 8)
    assert a > 0 and b > a and a % 256 == 0
    for bad in [pi.make_desc(4100, 16384, 128), pi.make_desc(4096, 16384, 12),
                pi.make_desc(4096, 0, 128), pi.make_desc(16384, 16384, 128),
                pi.make_desc(4096, 16384, 512)]:
        assert pi.pi_workspace_size(bad, 1) == 0
    bad = pi.make_desc(4096, 16384, 128)
    bad.dtype = 7
    assert pi.pi_workspace_size(bad, 1) == 0
    bad = pi.make_desc(4096, 16384, 128, hot_prefix=16385)
    assert pi.pi_workspace_size(bad, 1) == 0
    bad = pi.make_desc(4096, 16384, 128)
    bad.layout = 2
    assert pi.pi_workspace_size(bad, 1) == 0
    assert pi.pi_workspace_size(d, 0) == 0 and pi.pi_workspace_size(d, 33) == 0


def test_host_validation_before_launch(lib):
    # fake, aligned, never-dereferenced addresses: every call below fails
    # validation on the host and launches nothing
    P = 1 << 40
    d = pi.make_desc(1024, 4096, 64, "f16")
    w = pi.make_weights(P, P, P, P, P, None)
    ws_bytes = pi.pi_workspace_size(d, 1)
    L = lib
    by = ctypes.byref
    # NULL pointers
    assert L.pi_layer_decode(by(d), by(w), None, 1, P, None, None, None, P, P, ws_bytes,
                             None) == pi.PI_ERR_NULL
    assert L.pi_predict(by(d), None, P, P, P, 1, P, P, ws_bytes, None) == pi.PI_ERR_NULL
    assert L.pi_dense_ffn(None, by(w), P, 1, P, P, ws_bytes, None) == pi.PI_ERR_NULL
    # misalignment
    assert L.pi_layer_decode(by(d), by(w), P + 4, 1, P, None, None, None, P, P, ws_bytes,
                             None) == pi.PI_ERR_ALIGN
    w2 = pi.make_weights(P, P, P + 8, P, P, None)
    assert L.pi_sparse_ffn(by(d), by(w2), P, 1, P, P, 4096, None, None, None, P, P, P,
                           ws_bytes, None) == pi.PI_ERR_ALIGN
    # small workspace
    assert L.pi_layer_decode(by(d), by(w), P, 1, P, None, None, None, P, P, ws_bytes - 256,
                             None) == pi.PI_ERR_WORKSPACE
    # shapes / batch / dtype
    assert L.pi_layer_decode(by(d), by(w), P, 0, P, None, None, None, P, P, ws_bytes,
                             None) == pi.PI_ERR_SHAPE
    assert L.pi_predict(by(d), P, P, P, P, 33, P, P, ws_bytes, None) == pi.PI_ERR_SHAPE
    bad = pi.make_desc(1024, 4096, 64)
    bad.dtype = 3
    assert L.pi_dense_ffn(by(bad), by(w), P, 1, P, P, ws_bytes, None) == pi.PI_ERR_DTYPE
    assert L.pi_compact(P, 0, 1, P, P, 0, None, None, None, P, None, 0, None) == pi.PI_ERR_SHAPE
    assert L.pi_compact(P, 100, 1, P, P, 10, None, None, None, None, None, 0,
                        None) == pi.PI_ERR_NULL   # capacity may overflow: dev_status needed
    assert L.pi_compact(P, 100, 2, P, P, 100, P, None, P, P, None, 0,
                        None) == pi.PI_ERR_NULL   # union without its count
    # packed layout: W2 must be NULL; split layout: W2 required
    dp = pi.make_desc(1024, 4096, 64, "f16", packed=True)
    assert L.pi_layer_decode(by(dp), by(w), P, 1, P, None, None, None, P, P, ws_bytes,
                             None) == pi.PI_ERR_SHAPE
    w3 = pi.make_weights(P, P, P, P, None, None)
    assert L.pi_layer_decode(by(d), by(w3), P, 1, P, None, None, None, P, P, ws_bytes,
                             None) == pi.PI_ERR_NULL
    assert L.pi_pack_weights(by(d), P, None, P, None) == pi.PI_ERR_NULL
    assert L.pi_pack_weights(by(d), P + 2, P, P, None) == pi.PI_ERR_ALIGN
    assert L.pi_selftest_wait_timeout(P, P, 64, 1000000, None) == pi.PI_ERR_WORKSPACE
    assert L.pi_selftest_wait_timeout(P, P, 4096, 10, None) == pi.PI_ERR_SHAPE


def test_decode_layers_host_validation(lib):
    P = 1 << 40
    d = pi.make_desc(1024, 4096, 64, "f16", hot_prefix=90)
    w = pi.make_weights(P, P, P, P, P, None)
    wsb = pi.pi_workspace_size(d, 1)

    def f(*args):
        return pi.pi_decode_layers(*args, stream=0)  # the legacy stream: no torch.cuda here
    # layer count, step count, chain flag
    assert f([], [], 1, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_SHAPE
    assert f([d] * 129, [w] * 129, 1, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_SHAPE
    assert f([d], [w], 0, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_SHAPE
    assert f([d], [w], 4, P, 2, P, None, None, P, P, wsb) == pi.PI_ERR_SHAPE
    # layers of different shapes; hot prefixes and predictor ranks may differ,
    # with a workspace sized for the largest rank
    e = pi.make_desc(1024, 4096, 128, "f16")
    assert f([d, e], [w, w], 2, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_WORKSPACE
    assert pi.pi_workspace_size(e, 1) > wsb
    dd = pi.make_desc(2048, 4096, 64, "f16")
    assert f([d, dd], [w, w], 2, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_SHAPE
    g = pi.make_desc(1024, 4096, 64, "f16", gated=True)
    assert f([d, g], [w, w], 2, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_SHAPE
    # predictor weights required; NULL / misaligned buffers; small workspace
    wn = pi.make_weights(None, P, P, P, P, None)
    assert f([d], [wn], 1, P, 1, P, None, None, P, P, wsb) == pi.PI_ERR_NULL
    assert f([d], [w], 1, None, 1, P, None, None, P, P, wsb) == pi.PI_ERR_NULL
    assert f([d], [w], 1, P, 1, P, None, None, None, P, wsb) == pi.PI_ERR_NULL
    assert f([d], [w], 1, P + 4, 1, P, None, None, P, P, wsb) == pi.PI_ERR_ALIGN
    assert f([d], [w], 1, P, 1, P, P + 4, None, P, P, wsb) == pi.PI_ERR_ALIGN
    assert f([d], [w], 1, P, 1, P, None, None, P, P, wsb - 256) == pi.PI_ERR_WORKSPACE


def test_placement_host_validation(lib):
    P = 1 << 40
    L = lib
    by = ctypes.byref
    assert L.pi_profile_counts(P, 0, 1, P, None) == pi.PI_ERR_SHAPE
    assert L.pi_profile_counts(P, 10, 33, P, None) == pi.PI_ERR_SHAPE
    assert L.pi_profile_counts(None, 10, 1, P, None) == pi.PI_ERR_NULL
    assert L.pi_profile_counts(P, 10, 1, P + 4, None) == pi.PI_ERR_ALIGN
    assert L.pi_hot_order(P, 0, P, None) == pi.PI_ERR_SHAPE
    assert L.pi_hot_order(P, (1 << 22) + 1, P, None) == pi.PI_ERR_SHAPE
    assert L.pi_hot_order(P, 10, None, None) == pi.PI_ERR_NULL
    d = pi.make_desc(1024, 4096, 64, "f16")
    w = pi.make_weights(P, P, P, P, P, None)
    w2 = pi.make_weights(P + 4096, P, P + 8192, P + 16384, P + 32768, None)
    assert L.pi_permute_neurons(by(d), by(w), P, by(w2), None, None) == pi.PI_ERR_NULL
    assert L.pi_permute_neurons(by(d), by(w), None, by(w2), P, None) == pi.PI_ERR_NULL
    assert L.pi_permute_neurons(by(d), by(w), P + 4, by(w2), P, None) == pi.PI_ERR_ALIGN
    assert L.pi_permute_neurons(by(d), by(w), P, by(w), P, None) == pi.PI_ERR_SHAPE  # in place
    wbad = pi.make_weights(P, P, P, P, None, None)
    assert L.pi_permute_neurons(by(d), by(w), P, by(wbad), P, None) == pi.PI_ERR_NULL


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(pi, "_LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pi, "_lib", None)
    with pytest.raises(RuntimeError, match="libpi.so not found"):
        pi.lib()


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="addresses below are stand-ins: run only where no GPU is visible")
def test_static_scratch_rejects_shapes_beyond_its_size(lib):
    # n bytes of mask alone fill the fixed scratch: refused before any CUDA
    # call (no GPU exists here, so a CUDA call would have failed instead)
    n = pi.PI_STATIC_SCRATCH_BYTES
    desc = pi.make_desc(8192, n, 64, "f16")
    fake = 1 << 40  # never dereferenced: the call returns before launching
    w = pi.make_weights(fake, fake, fake, fake, fake, None)
    rc = pi.pi_layer_decode_static(desc, w, fake, fake, None, None, None, fake, stream=0)
    assert rc == pi.PI_ERR_WORKSPACE
