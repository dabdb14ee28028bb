"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/nvfp4kv.h declares, the host-only size queries match
the pages' byte accounting, and invalid arguments are rejected before any
CUDA call."""
import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nk():
    import __graft_entry__ as g
    from nvfp4_paged_kv_append_gb300 import build
    build.build()
    from nvfp4_paged_kv_append_gb300 import binding
    return binding


def header_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4kv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*((?:nvfp4|fp8)[a-z0-9_]*)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(nk):
    names = header_functions()
    assert len(names) >= 11, names
    for n in names:
        assert hasattr(nk.lib, n), n
    assert sorted(nk.EXPORTED) == names


def test_version_and_strings(nk):
    assert b"sm_103a" in nk.lib.nvfp4kv_version()
    assert nk.status_string(0) == "ok"
    assert "workspace" in nk.status_string(-3)


def test_cache_bytes_worked_examples(nk):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "accounting.json")))
    w = g["worked_per_token_L64"]
    assert w["layers"] * nk.nvfp4_cache_bytes(1, 1, w["kv_heads"], w["head_dim"]) == w["nvfp4_bytes_per_token"]
    w = g["worked_per_token_L80"]
    assert w["layers"] * nk.nvfp4_cache_bytes(1, 1, w["kv_heads"], w["head_dim"]) == w["nvfp4_bytes_per_token"]
    assert nk.nvfp4_cache_bytes(10, 16, 8, 128) == 10 * 16 * 8 * 144
    assert nk.nvfp4_cache_bytes(0, 16, 8, 128) == 0
    assert nk.nvfp4_cache_bytes(1, 16, 8, 100) == 0


def test_workspace_sizes(nk):
    # prefill: schedule items (8 B each) for every (q tile, kv head) + prefix
    b = nk.nvfp4_workspace_bytes(nk.OP_PREFILL, 1, 32, 8, 16384, 0)
    items = (16384 * 4 // 128 + 1) * 8
    assert b >= 16 + 8 * items and b % 16 == 0
    # decode: split partials (129 floats per split, head, request)
    d = nk.nvfp4_workspace_bytes(nk.OP_DECODE, 32, 32, 8, 0, 32768)
    # schedule: 16 B header + one 16 B record per (request, kv head, 1024-token split)
    assert d == 16 + 16 * 32 * 8 * 32 + 32 * 32 * 32 * 129 * 4
    assert nk.nvfp4_workspace_bytes(nk.OP_DECODE, 2, 6, 4, 0, 100) == 0  # Hq % Hkv != 0
    assert nk.nvfp4_workspace_bytes(7, 1, 8, 8, 1, 1) == 0


def test_invalid_arguments_rejected_on_host(nk):
    lib = nk.lib
    null = None
    # no cache descriptor
    assert lib.nvfp4_kv_append(null, null, null, 1, null, null) == -1
    d = nk.CacheDesc(16, 16, 32, 48, 4, 16, 2, 128, 1.0, 1.0)
    assert lib.nvfp4_kv_append(null, null, null, 1, ctypes.byref(d), null) == -1  # null k/v
    bad = nk.CacheDesc(16, 16, 32, 48, 4, 8, 2, 128, 1.0, 1.0)  # page_size 8
    assert lib.nvfp4_kv_append(null, null, null, 0, ctypes.byref(bad), null) == -1
    bad = nk.CacheDesc(17, 16, 32, 48, 4, 16, 2, 128, 1.0, 1.0)  # misaligned pool
    assert lib.nvfp4_kv_append(null, null, null, 0, ctypes.byref(bad), null) == -1
    bad = nk.CacheDesc(16, 16, 32, 48, 4, 16, 2, 128, 0.0, 1.0)  # zero scale
    assert lib.nvfp4_kv_append(null, null, null, 0, ctypes.byref(bad), null) == -1
    assert lib.nvfp4_kv_append(null, null, null, 0, ctypes.byref(d), null) == 0  # empty append is a no-op
    # prefill: Hq not a multiple of Hkv, bad variant, missing workspace
    args = lambda hq, variant, ws, qg=0.0: (16, 8, hq, ctypes.byref(d), 16, 1, 16, 16, 1, 1, 0.1, variant, qg, 16,
                                            null, ws, 64, null)
    assert lib.nvfp4_paged_prefill(*args(3, 0, 16)) == -1
    assert lib.nvfp4_paged_prefill(*args(6, 0, 16)) == -1   # ratio 3 is not a power of two
    assert lib.nvfp4_paged_prefill(*args(4, 3, 16)) == -1
    assert lib.nvfp4_paged_prefill(*args(4, 0, null)) == -3
    assert lib.nvfp4_paged_prefill(*args(4, 2, 16)) == -3   # FP4 PV needs room for its records
    assert lib.nvfp4_paged_prefill(*args(4, 0, 16, -1.0)) == -1          # query scale must be >= 0
    assert lib.nvfp4_paged_prefill(*args(4, 0, 16, float("nan"))) == -1  # and finite
    # decode: group of 32 unsupported; workspace too small
    assert lib.nvfp4_paged_decode(16, 64, ctypes.byref(d), 16, 1, 16, 1, 0.1, 16, null, 16, 16, null) == -1
    assert lib.nvfp4_paged_decode(16, 4, ctypes.byref(d), 16, 1, 16, 1, 0.1, 16, null, 16, 16, null) == -3
    # quantize: bad mode / non-positive global scale
    assert lib.nvfp4_quantize_rows(16, 1, 5, 1.0, 16, 16, null, null) == -1
    assert lib.nvfp4_quantize_rows(16, 1, 0, -1.0, 16, 16, null, null) == -1


def test_plan_run_and_noalloc_reject_bad_arguments_on_host(nk):
    """The split prefill entry points and the allocation-free one validate
    their arguments before touching the device, like nvfp4_paged_prefill."""
    lib = nk.lib
    null = None
    d = nk.CacheDesc(16, 16, 32, 48, 4, 16, 2, 128, 1.0, 1.0)
    plan = lambda hq, causal, variant, ws: lib.nvfp4_paged_prefill_plan(
        16, hq, ctypes.byref(d), 16, 1, 16, 16, 1, causal, variant, ws, 4096, null)
    assert plan(3, 1, 0, 16) == -1   # Hq not a multiple of Hkv
    assert plan(4, 2, 0, 16) == -1   # causal must be 0 or 1
    assert plan(4, 1, 7, 16) == -1   # unknown variant
    assert plan(4, 1, 0, null) == -3  # no workspace
    run = lambda q, scale: lib.nvfp4_paged_prefill_run(
        q, 16, 4, ctypes.byref(d), 16, 1, 16, 16, 1, 1, scale, 0, 0.0, 16, null, 16, 4096, null)
    assert run(16, float("nan")) == -1  # sm_scale must be finite
    assert run(8, 0.1) == -1            # q not 16-byte aligned
    assert run(null, 0.1) == -1         # no q
    noalloc = lambda hq: lib.nvfp4_paged_prefill_noalloc(
        16, 16, hq, ctypes.byref(d), 16, 1, 16, 16, 1, 1, 0.1, 0, 0.0, 16, null, null)
    assert noalloc(0) == -1
    assert noalloc(3) == -1


def test_token_major_rejects_bad_arguments_on_host(nk):
    """nvfp4_v_token_major checks its cache and buffers before any device
    work; an empty list is a no-op."""
    lib = nk.lib
    null = None
    d = nk.CacheDesc(16, 16, 32, 48, 4, 16, 2, 128, 1.0, 1.0)
    assert lib.nvfp4_v_token_major(null, 16, 1, 16, 16, null) == -1     # no cache
    assert lib.nvfp4_v_token_major(ctypes.byref(d), 16, -1, 16, 16, null) == -1
    assert lib.nvfp4_v_token_major(ctypes.byref(d), 16, 0, null, null, null) == 0
    assert lib.nvfp4_v_token_major(ctypes.byref(d), null, 1, 16, 16, null) == -1
    assert lib.nvfp4_v_token_major(ctypes.byref(d), 16, 1, 12, 16, null) == -1   # codes not 8-byte aligned
    bad = nk.CacheDesc(16, 16, 32, 48, 4, 16, 2, 64, 1.0, 1.0)                 # head_dim 64
    assert lib.nvfp4_v_token_major(ctypes.byref(bad), 16, 1, 16, 16, null) == -1


def test_header_and_library_from_plain_c(nk, tmp_path):
    """The boundary is a C ABI: a C99 program that includes the header and
    links the library calls the host-only entry points (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(nk.lib._name)
    src = tmp_path / "use_abi.c"
    src.write_text(
        "#include <stdio.h>\n#include <string.h>\n#include \"nvfp4kv.h\"\n"
        "int main(void) {\n"
        "  /* 144 B per token and kv head (K and V): one 16-token page of 8 heads */\n"
        "  if (nvfp4_cache_bytes(1, 16, 8, 128) != 16 * 8 * 144) return 1;\n"
        "  if (nvfp4_workspace_bytes(NVFP4KV_OP_PREFILL, 2, 6, 4, 0, 100) != 0) return 2;\n"
        "  if (strlen(nvfp4kv_version()) == 0) return 3;\n"
        "  if (nvfp4kv_status_string(NVFP4KV_ERR_SHAPE) == NULL) return 4;\n"
        "  printf(\"ok\\n\");\n  return 0;\n}\n")
    exe = tmp_path / "use_abi"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", str(src), "-I", os.path.join(root, "include"), "-L", libdir,
                    "-lnvfp4kv", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)


def test_fp8_host_entry_points(nk):
    """FP8 comparison cache: the pages' per-token byte figure and host-side
    argument checks (no GPU needed)."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "accounting.json")))["worked_per_token_L64"]
    assert g["layers"] * nk.fp8_cache_bytes(1, 1, g["kv_heads"], g["head_dim"]) == g["fp8_bytes_per_token"]
    lib = nk.lib
    null = None
    d = nk.Fp8CacheDesc(16, 32, 4, 16, 2, 128, 1.0, 1.0)
    assert lib.fp8_kv_append(null, null, null, 0, ctypes.byref(d), null) == 0     # empty append is a no-op
    assert lib.fp8_kv_append(null, null, null, 1, ctypes.byref(d), null) == -1    # null k/v
    bad = nk.Fp8CacheDesc(16, 32, 4, 16, 2, 128, 0.0, 1.0)                       # zero scale
    assert lib.fp8_kv_append(null, null, null, 0, ctypes.byref(bad), null) == -1
    bad = nk.Fp8CacheDesc(16, 40, 4, 16, 2, 128, 1.0, 1.0)                       # misaligned pool
    assert lib.fp8_kv_append(null, null, null, 0, ctypes.byref(bad), null) == -1
    # prefill needs room for the converted tiles
    ws_sched = nk.nvfp4_workspace_bytes(nk.OP_PREFILL, 1, 4, 2, 8, 0)
    assert nk.fp8_workspace_bytes(nk.OP_PREFILL, 1, 4, 2, 8, 16) == ws_sched + 2 * 65536
    assert nk.fp8_workspace_bytes(nk.OP_PREFILL, 1, 4, 2, 8, 0) == 0
    args = lambda hq, ws_bytes: (16, 8, hq, ctypes.byref(d), 16, 1, 16, 16, 1, 1, 0.1, 16, null, 16, ws_bytes, null)
    assert lib.fp8_paged_prefill(*args(3, 1 << 20)) == -1          # Hq not a multiple of Hkv
    assert lib.fp8_paged_prefill(*args(4, ws_sched)) == -3         # schedule only: no room for the tiles
    assert lib.fp8_paged_decode(16, 64, ctypes.byref(d), 16, 1, 16, 1, 0.1, 16, null, 16, 16, null) == -1
    assert lib.fp8_paged_decode(16, 4, ctypes.byref(d), 16, 1, 16, 1, 0.1, 16, null, 16, 16, null) == -3
