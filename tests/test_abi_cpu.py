"""The C ABI without a GPU: the library builds, loads, exports every declared symbol, and refuses
bad arguments with a status and a message before touching any device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mi_block.h")


@pytest.fixture(scope="module")
def lib():
    from diffusion_transformer_denoiser_gb300 import _build
    import diffusion_transformer_denoiser_gb300 as mi

    _build.build()
    return mi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set()
    for stmt in text.split(";"):
        stmt = stmt.strip()
        if stmt.startswith("typedef") or "(" not in stmt:
            continue
        m = re.search(r"\b(mi_[a-z0-9_]+)\s*\(", stmt)
        if m:
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mi_block_init", "mi_block_forward", "mi_denoise_step", "mi_block_workspace_size",
                     "mi_last_error", "mi_model_init"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib._name)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_version_and_message(lib):
    assert lib.mi_abi_version() == 1
    assert lib.mi_last_error() in (b"",) or isinstance(lib.mi_last_error(), bytes)


def _desc(mi, **kw):
    base = dict(hidden=256, n_heads=2, head_dim=128, mlp_inter=1024, eps=1e-6, fuse_epilogues=1,
                w_qkv=0x1000, w_o=0x2000, w_gu=0x3000, w_d=0x4000, q_norm_w=0x5000, k_norm_w=0x6000)
    base.update(kw)
    return mi._BlockDesc(**base)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(head_dim=64), 2, "head_dim"),
    (dict(hidden=384, n_heads=3), 2, "multiple of 256"),
    (dict(hidden=512), 1, "n_heads"),
    (dict(mlp_inter=1000), 2, "mlp_inter"),
    (dict(w_o=0), 1, "w_o is null"),
    (dict(w_gu=0x3008), 1, "16-byte aligned"),
])
def test_block_init_refusals(lib, kw, status, needle):
    import diffusion_transformer_denoiser_gb300 as mi

    d = _desc(mi, **kw)
    h = ctypes.c_void_p()
    st = lib.mi_block_init(ctypes.byref(h), ctypes.byref(d))
    assert st == status
    assert needle in lib.mi_last_error().decode()
    assert not h.value


def test_null_arguments(lib):
    assert lib.mi_block_init(None, None) == 1
    assert lib.mi_block_forward(None, None, None, None, None, None, None, 0, None, None, 0, None) == 1
    assert lib.mi_gemm_bf16(None, None, None, 4, 8, 64, None) == 1
    assert lib.mi_model_plan(None, None, 1, 0, None, None) == 1


def test_gemm_shape_refusal(lib):
    # fake aligned pointers: the shape is refused before any device work
    assert lib.mi_gemm_bf16(0x1000, 0x2000, 0x3000, 16, 8, 100, None) == 2
    assert "multiple of 64" in lib.mi_last_error().decode()
    assert lib.mi_gemm_bf16(0x1000, 0x2000, 0x3000, 16, 12, 64, None) == 2
    assert lib.mi_gemm_bf16_silu_gate(0x1000, 0x2000, 0x3000, 16, 64, 64, None) == 2


def test_no_device_is_an_error_not_a_crash(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.mi_device_supported() != 0


def test_product_path_does_not_import_the_oracle():
    # the CUDA binding and build never reference the oracle package
    pkg = os.path.join(ROOT, "diffusion_transformer_denoiser_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("oracle is", ""), f
