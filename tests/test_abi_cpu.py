"""The C-ABI library loads without a GPU and exports every entry point that
include/h3dit.h declares; the Python binding names each of them.  No compute
call is made here."""
import ctypes
import os
import re

import pytest

from audio_diffusion_transformer_fwd_b300 import build as B
from audio_diffusion_transformer_fwd_b300 import h3dit as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "h3dit.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(h3dit_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ctypes.CDLL(B.LIB)


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert len(syms) >= 20
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in h3dit.h but not exported"


def test_binding_covers_the_header():
    assert sorted(H._EXPORTS) == declared_symbols()


def test_host_only_calls(lib):
    lib.h3dit_version.restype = ctypes.c_int
    assert lib.h3dit_version() == 2
    g = H.video_grid(0, 6, 30, 54)
    assert H.lib().h3dit_reduced_tokens(10488, ctypes.byref(g)) == 5628
    bad = H.video_grid(0, 6, 30, 54)
    assert H.lib().h3dit_reduced_tokens(100, ctypes.byref(bad)) == -1
    shape = H.BlockShape(5120, 40, 128, 20480)
    n1 = H.h3dit_workspace_size(shape, 6912)
    n2 = H.h3dit_workspace_size(shape, 10488)
    n3 = H.h3dit_workspace_size(shape, 10488, H.reduction(g, 3, 40))
    assert 0 < n1 < n2 < n3
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_workspace_size(H.BlockShape(5120, 40, 96, 20480), 10)
    assert e.value.status == H.E_INVAL
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_workspace_size(H.BlockShape(5120, 80, 64, 20000), 10)
    assert e.value.status == H.E_UNSUPPORTED
    assert "ffn" in H.lib().h3dit_last_error().decode()


def test_int8_shape_checks_on_host():
    w = (256, 4, 64)
    ok = H.BlockShape(*w, 1024, precision=H.INT8, rope_sections=(16, 24, 24))
    assert H.h3dit_workspace_size(ok, 16) > H.h3dit_workspace_size(
        H.BlockShape(*w, 1024, rope_sections=(16, 24, 24)), 16)
    bad = H.BlockShape(*w, 1280, precision=H.INT8, rope_sections=(16, 24, 24))
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_workspace_size(bad, 16)
    assert e.value.status == H.E_UNSUPPORTED
    # the same ffn is fine in BF16
    H.h3dit_workspace_size(H.BlockShape(*w, 1280, rope_sections=(16, 24, 24)), 16)


def test_workspace_aliasing_saves_memory():
    """Arena aliasing keeps the block's activations to roughly
    max(3Nd + V^T padding, NF) + 2Nd BF16 values plus the RoPE table."""
    shape = H.BlockShape(5120, 40, 128, 20480)
    n = 10488
    got = H.h3dit_workspace_size(shape, n)
    unaliased = 2 * n * (5120 * (1 + 3 + 1 + 1 + 1 + 1) + 20480)   # h, qkv, o, a, h2, m, u
    assert got < 0.8 * unaliased


@pytest.mark.parametrize("fault,status,word", [("alloc", H.E_NOMEM, "workspace"), ("arg", H.E_INVAL, "argument"),
                                               ("shape", H.E_UNSUPPORTED, "shape"), ("launch", H.E_CUDA, "launch")])
def test_injected_faults_reach_the_caller(lib, monkeypatch, fault, status, word):
    """H3DIT_FAULT makes the block and step entry points fail where that
    failure would arise, before anything is enqueued (no GPU is needed: the
    pointers below are never dereferenced)."""
    shape = H.BlockShape(256, 4, 64, 1024, 1e-6, (16, 24, 24))
    fake = 1 << 20                                   # aligned, never dereferenced
    bw = H.block_weights(fake, fake, fake, fake)
    n = 256
    need = H.h3dit_workspace_size(shape, n)
    g = H.video_grid(0, 2, 8, 12)
    tr = H.reduction(g, 0, 1)
    need_tr = H.h3dit_workspace_size(shape, n, tr)
    monkeypatch.setenv("H3DIT_FAULT", fault)
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward(shape, bw, fake, fake, fake, n, fake, need, stream=0)
    assert e.value.status == status and word in str(e.value) and "H3DIT_FAULT" in str(e.value)
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_step_forward(shape, [bw, bw], fake, fake, fake, n, tr, fake, need_tr, stream=0)
    assert e.value.status == status and "H3DIT_FAULT" in str(e.value)
    # genuine argument errors still win over an injected allocation failure
    if fault == "alloc":
        with pytest.raises(H.H3DitError) as e:
            H.h3dit_block_forward(shape, bw, fake, None, fake, n, fake, need, stream=0)
        assert e.value.status == H.E_INVAL
    monkeypatch.delenv("H3DIT_FAULT")
    # a short workspace is refused without any injection
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward(shape, bw, fake, fake, fake, n, fake, need - 256, stream=0)
    assert e.value.status == H.E_NOMEM


def test_stall_request_arguments(lib):
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_test_stall_next_gemm(-2)
    assert e.value.status == H.E_INVAL
    H.h3dit_test_stall_next_gemm(-1)


def test_int8_weight_bytes_checked_on_host(lib):
    """codes_int8 must be 0 or 1, and int8 weight bytes 8-byte aligned; both
    are refused before anything is enqueued."""
    shape = H.BlockShape(256, 4, 64, 1024, 1e-6, (16, 24, 24), precision=H.INT8)
    fake = 1 << 20
    n = 256
    need = H.h3dit_workspace_size(shape, n)
    assert need > H.h3dit_workspace_size(H.BlockShape(256, 4, 64, 1024, 1e-6, (16, 24, 24)), n)
    bad = H.block_weights(fake + 4, fake, fake, fake, fake, fake, fake, fake, codes_int8=True)
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward(shape, bad, fake, fake, fake, n, fake, need, stream=0)
    assert e.value.status == H.E_INVAL and "aligned" in str(e.value)
    odd = H.block_weights(fake, fake, fake, fake, fake, fake, fake, fake)
    odd.codes_int8 = 2
    with pytest.raises(H.H3DitError) as e:
        H.h3dit_block_forward(shape, odd, fake, fake, fake, n, fake, need, stream=0)
    assert e.value.status == H.E_INVAL and "codes_int8" in str(e.value)
