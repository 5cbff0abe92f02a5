"""The C ABI on the host: the library loads, exports every declared symbol,
validates shapes in prepare (no GPU needed) and reports errors."""

import ctypes
import os
import re

import pytest

import datagen
import fusion_backend_gb300 as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fb.build()
    return fb.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_ffn_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fb.EXPORTS)


def test_prepare_reports_workspace_without_device(lib):
    plan, ws = fb.moe_ffn_prepare(datagen.Shapes(1, 2048, 128, 8, 768, 512), fb.ACT_BF16, fb.W_BF16)
    assert ws > 0 and ws % 256 == 0
    assert fb.moe_ffn_query(plan, fb.QUERY_PATH) == 0
    assert fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE) == 1
    fb.moe_ffn_destroy(plan)


@pytest.mark.parametrize(
    "shapes,wfmt",
    [
        (datagen.Shapes(0, 256, 8, 2, 128, 256), fb.W_BF16),      # T = 0
        (datagen.Shapes(1, 260, 8, 2, 128, 256), fb.W_BF16),      # H not a multiple of 8
        (datagen.Shapes(1, 256, 8, 9, 128, 256), fb.W_BF16),      # top_k > E
        (datagen.Shapes(1, 256, 40, 33, 128, 256), fb.W_BF16),    # top_k > 32
        (datagen.Shapes(1, 256, 2000, 2, 128, 256), fb.W_BF16),   # E > 1024
        (datagen.Shapes(1, 264, 8, 2, 128, 256), fb.W_Q4B32),     # 4-bit rows need H a multiple of 256
        (datagen.Shapes(1, 8192, 8, 2, 128, 256), fb.W_BF16),     # H > 4096 (decode path bound)
        (datagen.Shapes(9, 256, 8, 2, 192, 256), fb.W_Q4B32),     # T > 8, 4-bit: I a multiple of 128
        (datagen.Shapes(1025, 256, 8, 2, 128, 256), fb.W_BF16),   # T > 1024
        (datagen.Shapes(64, 128, 8, 2, 128, 256), fb.W_BF16),     # T > 8: H a multiple of 256
        (datagen.Shapes(64, 256, 8, 2, 192, 256), fb.W_BF16),     # T > 8: I a multiple of 128
        (datagen.Shapes(64, 256, 300, 2, 128, 256), fb.W_BF16),   # T > 8: E <= 256
        (datagen.Shapes(1, 264, 8, 2, 128, 256), fb.W_I8),        # int8 rows need H a multiple of 16
        (datagen.Shapes(64, 256, 8, 2, 128, 256), fb.W_I8),       # int8 weights: decode path only
    ],
)
def test_prepare_rejects_unsupported(lib, shapes, wfmt):
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_prepare(shapes, fb.ACT_BF16, wfmt)
    assert e.value.status == fb.ERR_UNSUPPORTED


def test_batched_path_needs_bf16_activation(lib):
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_prepare(datagen.Shapes(64, 256, 8, 2, 128, 256), fb.ACT_F32, fb.W_BF16)
    assert e.value.status == fb.ERR_UNSUPPORTED


def test_prepare_batched_plan_and_workspace(lib):
    s = datagen.Shapes(256, 2048, 128, 8, 768, 512)
    plan, ws = fb.moe_ffn_prepare(s, fb.ACT_BF16, fb.W_BF16)
    assert fb.moe_ffn_query(plan, fb.QUERY_PATH) == 1
    assert fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE) == 6
    TK = s.T * s.top_k
    # at least x by slot (bf16), h by slot (bf16) and y by slot (fp32)
    assert ws >= TK * s.H * 2 + (TK + s.T) * s.I * 2 + (TK + s.T) * s.H * 4
    fb.moe_ffn_destroy(plan)


def test_prepare_batched_q4_plan_and_workspace(lib):
    s = datagen.Shapes(64, 2048, 128, 8, 768, 512)
    plan, ws = fb.moe_ffn_prepare(s, fb.ACT_BF16, fb.W_Q4B32)
    assert fb.moe_ffn_query(plan, fb.QUERY_PATH) == 1
    assert fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE) == 6
    TK = s.T * s.top_k
    # x by slot incl. the shared slots (fp16), h by slot (fp16), y by slot (fp32)
    assert ws >= (TK + s.T) * s.H * 2 + (TK + s.T) * s.I * 2 + (TK + s.T) * s.H * 4
    fb.moe_ffn_destroy(plan)


def test_prepare_int8_decode_plan(lib):
    for s in (datagen.Shapes(1, 2048, 128, 8, 768, 512), datagen.Shapes(8, 272, 8, 2, 130, 70)):
        plan, ws = fb.moe_ffn_prepare(s, fb.ACT_BF16, fb.W_I8)
        assert ws > 0 and ws % 256 == 0
        assert fb.moe_ffn_query(plan, fb.QUERY_PATH) == 0
        assert fb.moe_ffn_query(plan, fb.QUERY_LAUNCHES_PER_EXECUTE) == 1
        fb.moe_ffn_destroy(plan)


def test_prepare_rejects_bad_enums_and_nulls(lib):
    s = fb.Shapes(1, 256, 8, 2, 128, 256)
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    assert lib.moe_ffn_prepare(ctypes.byref(s), fb.DType(5, 0), ctypes.byref(plan), ctypes.byref(ws)) == fb.ERR_INVALID_ARG
    assert lib.moe_ffn_prepare(ctypes.byref(s), fb.DType(0, 7), ctypes.byref(plan), ctypes.byref(ws)) == fb.ERR_INVALID_ARG
    assert lib.moe_ffn_prepare(None, fb.DType(0, 0), ctypes.byref(plan), ctypes.byref(ws)) == fb.ERR_INVALID_ARG


def test_execute_argument_errors_before_any_device_call(lib):
    plan, ws = fb.moe_ffn_prepare(datagen.Shapes(1, 256, 8, 2, 128, 256), fb.ACT_F32, fb.W_BF16)
    fake = 1 << 20  # aligned, never dereferenced: validation fails first
    # null plan / null pointers
    assert lib.moe_ffn_execute(None, None, fake, ws, fake, fake, fake, fake, fake, fake) == fb.ERR_INVALID_ARG
    assert lib.moe_ffn_execute(plan, None, fake, ws, None, fake, fake, fake, fake, fake) == fb.ERR_INVALID_ARG
    # workspace too small
    assert lib.moe_ffn_execute(plan, None, fake, ws - 1, fake, fake, fake, fake, fake, fake) == fb.ERR_WORKSPACE
    # misaligned
    assert lib.moe_ffn_execute(plan, None, fake + 8, ws, fake, fake, fake, fake, fake, fake) == fb.ERR_MISALIGNED
    assert lib.moe_ffn_execute(plan, None, fake, ws, fake + 4, fake, fake, fake, fake, fake) == fb.ERR_MISALIGNED
    # block form needs a bf16-activation plan
    assert lib.moe_ffn_execute_block(plan, None, fake, ws, fake, fake, fake, fake, fake, 1e-6, None, None) == fb.ERR_UNSUPPORTED
    assert lib.moe_ffn_execute_block(plan, None, fake, ws, fake, fake, fake, fake, fake, -1.0, None, None) == fb.ERR_INVALID_ARG
    fb.moe_ffn_destroy(plan)


def test_strerror_covers_codes(lib):
    for code in range(0, -8, -1):
        assert fb.strerror(code) != "unknown status"
    assert fb.strerror(-99) == "unknown status"


def test_two_stream_workspace_query(lib):
    plan, ws = fb.moe_ffn_prepare(datagen.Shapes(1, 2048, 128, 8, 768, 512), fb.ACT_BF16, fb.W_BF16)
    two = fb.moe_ffn_query(plan, fb.QUERY_TWO_STREAM_WORKSPACE)
    # both branches' own workspaces, then their two [T][H] fp32 outputs
    assert two == 2 * ws + 2 * 2048 * 4
    fb.moe_ffn_destroy(plan)
    plan, _ = fb.moe_ffn_prepare(datagen.Shapes(64, 2048, 128, 8, 768, 512), fb.ACT_BF16, fb.W_BF16)
    with pytest.raises(fb.MoeFFNError) as e:
        fb.moe_ffn_query(plan, fb.QUERY_TWO_STREAM_WORKSPACE)
    assert e.value.status == fb.ERR_UNSUPPORTED
    fb.moe_ffn_destroy(plan)


def test_missing_library_fails_loudly(tmp_path):
    """No CPU fallback: without the built library every entry of the binding raises, naming the file."""
    import subprocess
    import sys

    code = (
        "import fusion_backend_gb300 as fb\n"
        f"fb.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
        "try:\n"
        "    fb.moe_ffn_prepare(fb.Shapes(1, 256, 8, 2, 128, 256), fb.ACT_F32, fb.W_BF16)\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('no error')\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "raised:" in r.stdout and "absent.so" in r.stdout, r.stdout
