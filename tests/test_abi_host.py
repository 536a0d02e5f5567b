"""Host-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every function include/pa.h declares, and rejects bad arguments before any
CUDA call.  No GPU is needed (no compute entry point reaches a launch here)."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_attention_14_gb300 import build as pa_build
from paged_kv_attention_14_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    path = pa_build.build()
    return B.load(path)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary_entry_points():
    names = _declared_functions()
    for want in ("pa_cache_write", "pa_decode", "pa_prefill_chunk", "pa_merge_partials"):
        assert want in names
    assert set(names) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(pa_[a-z_0-9]+)$", out, flags=re.M))
    declared = set(_declared_functions())
    assert declared <= exported, declared - exported
    # nothing else leaks out of the library under the pa_ prefix
    assert exported == declared


def test_abi_version(lib):
    assert lib.pa_abi_version() == B.ABI_VERSION == 4
    m = re.search(r"#define\s+PA_ABI_VERSION\s+(\d+)", open(HEADER).read())
    assert int(m.group(1)) == lib.pa_abi_version()


def test_desc_struct_matches_header_layout():
    # field order of pa_kv_desc in the header
    text = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} pa_kv_desc;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b(\w+);", body)
    assert fields == [f for f, _ in B.PaKvDesc._fields_]
    assert ctypes.sizeof(B.PaKvDesc) == 80


def _desc(**kw):
    d = dict(num_blocks=64, num_kv_heads=2, num_q_heads=4, head_dim=64)
    d.update(kw)
    return B.make_desc(**d)


def test_cache_write_argument_errors(lib):
    null = None
    d = _desc()
    # NULL descriptor
    assert lib.pa_cache_write(None, null, null, null, null, null, 4, null) == B.PA_ERR_INVALID_ARG
    assert "desc" in B.last_error()
    # zero tokens is a no-op
    assert lib.pa_cache_write(ctypes.byref(d), null, null, null, null, null, 0, null) == B.PA_OK
    assert B.last_error() == ""
    # NULL pointers
    assert lib.pa_cache_write(ctypes.byref(d), null, null, null, null, null, 4, null) == B.PA_ERR_INVALID_ARG
    # misaligned
    assert lib.pa_cache_write(ctypes.byref(d), 0x1008, 0x2000, 0x3000, 0x4000, 0x5000, 4, null) == B.PA_ERR_INVALID_ARG
    assert "aligned" in B.last_error()
    # negative count
    assert lib.pa_cache_write(ctypes.byref(d), 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, -1, null) == B.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value,status", [
    ("block_size", 32, B.PA_ERR_UNSUPPORTED),
    ("head_dim", 96, B.PA_ERR_UNSUPPORTED),
    ("num_q_heads", 5, B.PA_ERR_INVALID_ARG),     # not a multiple of 2 kv heads
    ("num_kv_heads", 0, B.PA_ERR_INVALID_ARG),
    ("num_q_heads", 34, B.PA_ERR_UNSUPPORTED),    # group size 17
    ("kv_dtype", 7, B.PA_ERR_INVALID_ARG),
    ("num_blocks", -1, B.PA_ERR_INVALID_ARG),
    ("sliding_window", -1, B.PA_ERR_INVALID_ARG),
    ("attention_chunk", -5, B.PA_ERR_INVALID_ARG),
])
def test_descriptor_validation(lib, field, value, status):
    d = _desc()
    setattr(d, field, value)
    if field == "num_q_heads" and value == 34:
        d.num_kv_heads = 2
    got = lib.pa_decode(ctypes.byref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 2, 16,
                        0.125, 0x7000, 1 << 20, None)
    assert got == status, B.last_error()
    assert B.last_error() != ""


def test_fp8_scales_must_be_non_negative(lib):
    d = _desc(kv_dtype=B.PA_KV_FP8_E4M3, k_scale=-1.0)
    assert lib.pa_cache_write(ctypes.byref(d), 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, None) == B.PA_ERR_INVALID_ARG
    d = _desc(kv_dtype=B.PA_KV_FP8_E4M3, k_scale=float("nan"))
    assert lib.pa_cache_write(ctypes.byref(d), 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, None) == B.PA_ERR_INVALID_ARG


def test_fp16_cache_is_accepted_and_ignores_scales(lib):
    # 16-bit caches take no scales: a negative one is not an error there
    for kv in (B.PA_KV_F16, B.PA_KV_BF16):
        d = _desc(kv_dtype=kv, k_scale=-1.0, v_scale=-2.0)
        assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_OK, B.last_error()
    d = _desc(kv_dtype=B.PA_KV_F16 + 1)
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_ERR_INVALID_ARG


def test_per_head_scales_only_with_fp8_and_aligned(lib):
    d = _desc(kv_dtype=B.PA_KV_BF16)
    d.k_scales = 0x1000
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_ERR_INVALID_ARG
    assert "FP8" in B.last_error()
    d = _desc(kv_dtype=B.PA_KV_FP8_E4M3)
    d.v_scales = 0x1002
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_ERR_INVALID_ARG
    assert "aligned" in B.last_error()
    d.v_scales = 0x1004
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_OK


def test_prefix_attention_and_copy_blocks_argument_errors(lib):
    d = _desc()
    P = ctypes.c_void_p
    ok = (0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000)
    # nothing to do
    assert lib.pa_prefix_attention(ctypes.byref(d), *ok[:2], 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 4, 0x8000,
                                   0, 16, 64, 1, 0, 0.1, None) == B.PA_OK
    # lse is required
    assert lib.pa_prefix_attention(ctypes.byref(d), 0x1000, None, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 4,
                                   0x8000, 2, 16, 64, 1, 0, 0.1, None) == B.PA_ERR_INVALID_ARG
    # prefix longer than its table
    assert lib.pa_prefix_attention(ctypes.byref(d), *ok[:2], 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 4, 0x8000,
                                   2, 16, 65, 1, 0, 0.1, None) == B.PA_ERR_INVALID_ARG
    # zero splits, or fewer slots than splits
    assert lib.pa_prefix_attention(ctypes.byref(d), *ok[:2], 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 4, 0x8000,
                                   2, 16, 64, 0, 0, 0.1, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_prefix_attention(ctypes.byref(d), *ok[:2], 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 4, 0x8000,
                                   2, 16, 64, 3, 2, 0.1, None) == B.PA_ERR_INVALID_ARG
    # local attention does not apply to a shared prefix
    dw = _desc(sliding_window=8)
    assert lib.pa_prefix_attention(ctypes.byref(dw), *ok[:2], 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 4, 0x8000,
                                   2, 16, 64, 1, 0, 0.1, None) == B.PA_ERR_UNSUPPORTED
    # block copies: none to do; NULL arrays; misaligned cache
    assert lib.pa_copy_blocks(ctypes.byref(d), None, None, None, None, 0, None) == B.PA_OK
    assert lib.pa_copy_blocks(ctypes.byref(d), 0x1000, 0x2000, None, 0x3000, 3, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(ctypes.byref(d), 0x1008, 0x2000, 0x3000, 0x4000, 3, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(ctypes.byref(d), 0x1000, 0x2000, 0x3002, 0x4000, 3, None) == B.PA_ERR_INVALID_ARG


def test_prefill_sequence_count_limit(lib):
    d = _desc()
    # more sequences than one grid dimension holds: rejected before any launch
    assert lib.pa_prefill_chunk(ctypes.byref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 4, 0x7000,
                                70000, 16, 64, 0.1, None) == B.PA_ERR_UNSUPPORTED
    assert "65535" in B.last_error()


def test_decode_argument_errors(lib):
    d = _desc()
    ok_ptrs = (0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000)
    # zero sequences: nothing to do
    assert lib.pa_decode(ctypes.byref(d), *ok_ptrs, 4, 0x6000, 0, 16, 0.1, None, 0, None) == B.PA_OK
    # NULL out
    assert lib.pa_decode(ctypes.byref(d), None, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 2, 16, 0.1,
                         0x7000, 1 << 20, None) == B.PA_ERR_INVALID_ARG
    # max_context_len beyond the table
    assert lib.pa_decode(ctypes.byref(d), *ok_ptrs, 4, 0x6000, 2, 65, 0.1, 0x7000, 1 << 20,
                         None) == B.PA_ERR_INVALID_ARG
    # NaN scale
    assert lib.pa_decode(ctypes.byref(d), *ok_ptrs, 4, 0x6000, 2, 16, float("nan"), 0x7000, 1 << 20,
                         None) == B.PA_ERR_INVALID_ARG
    # misaligned block table
    assert lib.pa_decode(ctypes.byref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5002, 4, 0x6000, 2, 16, 0.1,
                         0x7000, 1 << 20, None) == B.PA_ERR_INVALID_ARG
    # unknown decode kernel
    d2 = _desc(decode_impl=9)
    assert lib.pa_decode(ctypes.byref(d2), *ok_ptrs, 4, 0x6000, 2, 16, 0.1, 0x7000, 1 << 20,
                         None) == B.PA_ERR_INVALID_ARG


def test_decode_append_argument_errors(lib):
    # the checks that need no device run before anything is planned or enqueued
    d = _desc()
    ptrs = (0x1000, None, 0x2000)          # out, lse, q
    caches = (0x3000, 0x4000, 0x5000, 4, 0x6000)  # k_cache, v_cache, block_tables, width, context_lens
    # zero sequences: nothing to do, k_new / v_new not needed
    assert lib.pa_decode_append(ctypes.byref(d), *ptrs, None, None, *caches, 0, 16, 0.1, None, 0, None) == B.PA_OK
    # k_new / v_new NULL or misaligned
    assert lib.pa_decode_append(ctypes.byref(d), *ptrs, None, 0x8000, *caches, 2, 16, 0.1, 0x7000, 1 << 20,
                                None) == B.PA_ERR_INVALID_ARG
    assert "k_new" in B.last_error()
    assert lib.pa_decode_append(ctypes.byref(d), *ptrs, 0x8000, 0x9008, *caches, 2, 16, 0.1, 0x7000, 1 << 20,
                                None) == B.PA_ERR_INVALID_ARG
    # an 8-bit cache's descriptor is checked as pa_decode checks it (a negative scale)
    d8 = _desc(kv_dtype=B.PA_KV_FP8_E4M3, k_scale=-1.0, v_scale=1.0)
    assert lib.pa_decode_append(ctypes.byref(d8), *ptrs, 0x8000, 0x9000, *caches, 2, 16, 0.1, 0x7000, 1 << 20,
                                None) == B.PA_ERR_INVALID_ARG
    # pa_decode's own checks: NULL out, a length beyond the table, a bad descriptor
    assert lib.pa_decode_append(ctypes.byref(d), None, None, 0x2000, 0x8000, 0x9000, *caches, 2, 16, 0.1, 0x7000,
                                1 << 20, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_decode_append(ctypes.byref(d), *ptrs, 0x8000, 0x9000, *caches, 2, 65, 0.1, 0x7000, 1 << 20,
                                None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_decode_append(ctypes.byref(_desc(head_dim=96)), *ptrs, 0x8000, 0x9000, *caches, 2, 16, 0.1,
                                0x7000, 1 << 20, None) == B.PA_ERR_UNSUPPORTED


def test_error_word_and_check_flag_validation(lib):
    d = _desc()
    d.error_word = 0x1002  # not 4-byte aligned
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_ERR_INVALID_ARG
    assert "error_word" in B.last_error()
    d.error_word = 0x1004
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_OK
    d.check_indices = 2
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_ERR_INVALID_ARG
    assert "check_indices" in B.last_error()
    d.check_indices = 1
    assert lib.pa_cache_write(ctypes.byref(d), None, None, None, None, None, 0, None) == B.PA_OK


def test_stall_hook_arguments(lib):
    assert lib.pa_test_stall_pipelines(1, 0) == B.PA_ERR_INVALID_ARG
    assert lib.pa_test_stall_pipelines(1, -5) == B.PA_ERR_INVALID_ARG
    assert lib.pa_test_stall_pipelines(0, 0) == B.PA_OK


def test_static_decode_checks_arguments_like_pa_decode(lib):
    # an argument error is reported with pa_decode's status, before anything
    # is enqueued (no GPU is touched here)
    assert lib.pa_decode_static(None, 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 2, 16, 0.1,
                                None) == B.PA_ERR_INVALID_ARG
    d = _desc(head_dim=96)
    assert lib.pa_decode_static(ctypes.byref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 2, 16,
                                0.1, None) == B.PA_ERR_UNSUPPORTED
    d = _desc()
    assert lib.pa_decode_static(ctypes.byref(d), None, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 2, 16,
                                0.1, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_decode_static(ctypes.byref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 2, 65,
                                0.1, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_decode_static(ctypes.byref(d), 0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 4, 0x6000, 0, 16,
                                0.1, None) == B.PA_OK


def test_mixed_attention_argument_errors(lib):
    d = _desc()
    assert lib.pa_mixed_workspace_size(None, 4, 16) == 0
    null = None
    args = (null, null, null, null, 4, null, 0, 0, null, null, null, null, null, 4, null, 0, 0, 0, 0x3000, 0x4000,
            0.1, 0x7000, 1 << 20, null)
    assert lib.pa_mixed_attention(None, *args) == B.PA_ERR_INVALID_ARG
    # a decode part with a NULL output
    bad = (null, null, 0x2000, 0x5000, 4, 0x6000, 2, 16) + args[8:]
    assert lib.pa_mixed_attention(ctypes.byref(d), *bad) == B.PA_ERR_INVALID_ARG
    # an unsupported cache type for the single launch (head_dim 64) is refused on the host
    assert B.last_error() != ""


def test_prefill_argument_errors(lib):
    d = _desc()
    args = (0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 4, 0x7000)
    assert lib.pa_prefill_chunk(ctypes.byref(d), *args, 0, 8, 16, 0.1, None) == B.PA_OK
    assert lib.pa_prefill_chunk(ctypes.byref(d), None, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 4, 0x7000,
                                2, 8, 16, 0.1, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_prefill_chunk(ctypes.byref(d), *args, 2, 8, 100, 0.1, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_prefill_chunk(ctypes.byref(d), 0x1004, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 4, 0x7000,
                                2, 8, 16, 0.1, None) == B.PA_ERR_INVALID_ARG


def test_balanced_prefill_argument_errors(lib):
    d = _desc()
    args = (0x1000, None, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 4, 0x7000)
    # nothing to do: no workspace needed
    assert lib.pa_prefill_chunk_balanced(ctypes.byref(d), *args, 0, 8, 16, 0.1, None, 0, None) == B.PA_OK
    # the workspace is required, 16-byte aligned, and checked after the other arguments
    assert lib.pa_prefill_chunk_balanced(ctypes.byref(d), *args, 2, 8, 16, 0.1, None, 1 << 20,
                                         None) == B.PA_ERR_WORKSPACE
    assert lib.pa_prefill_chunk_balanced(ctypes.byref(d), *args, 2, 8, 16, 0.1, 0x8008, 1 << 20,
                                         None) == B.PA_ERR_WORKSPACE
    assert lib.pa_prefill_chunk_balanced(ctypes.byref(d), *args, 2, 8, 100, 0.1, None, 0,
                                         None) == B.PA_ERR_INVALID_ARG
    # the schedule query and the sizes reject invalid descriptors; an empty batch runs nothing
    bad = _desc(head_dim=96)
    assert lib.pa_prefill_balanced_chosen(ctypes.byref(bad), 2, 8, 16, 4) == -1
    assert lib.pa_prefill_workspace_size(ctypes.byref(bad), 2, 8) == 0
    assert lib.pa_prefill_balanced_chosen(ctypes.byref(d), 0, 8, 16, 4) == 0
    assert lib.pa_prefill_balanced_chosen(ctypes.byref(d), 2, 8, -1, 4) == -1
    # the test hook takes 0, 1 or 2
    assert lib.pa_test_prefill_schedule(3) == B.PA_ERR_INVALID_ARG
    assert lib.pa_test_prefill_schedule(0) == B.PA_OK


def test_merge_argument_errors(lib):
    assert lib.pa_merge_partials(0x1000, None, 0x2000, 0x3000, None, 0, 4, 2, 64, None) == B.PA_OK
    assert lib.pa_merge_partials(0x1000, None, 0x2000, 0x3000, None, 2, 4, 2, 66, None) == B.PA_ERR_UNSUPPORTED
    assert lib.pa_merge_partials(None, None, 0x2000, 0x3000, None, 2, 4, 2, 64, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_merge_partials(0x1000, None, 0x2000, 0x3000, None, 2, 0, 2, 64, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_merge_partials(0x1000, None, 0x2008, 0x3000, None, 2, 4, 2, 64, None) == B.PA_ERR_INVALID_ARG


def test_last_error_is_per_thread(lib):
    import threading
    assert lib.pa_cache_write(None, None, None, None, None, None, 1, None) == B.PA_ERR_INVALID_ARG
    seen = []
    t = threading.Thread(target=lambda: seen.append(B.last_error()))
    t.start()
    t.join()
    assert seen == [""]
    assert B.last_error() != ""


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        B.load(str(tmp_path / "nope.so"))


def test_header_is_valid_c_and_links_every_entry_point(tmp_path):
    """A C99 caller: pa.h compiles with -Wall -Wextra -Werror, every declared
    entry point links against the library, and the descriptor's size and field
    offsets seen from C match the binding's."""
    import shutil
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    names = _declared_functions()
    fields = [f for f, _ in B.PaKvDesc._fields_]
    src = tmp_path / "caller.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"pa.h\"\n"
        "int main(void) {\n"
        "  void (*fns[])(void) = {" + ", ".join(f"(void (*)(void)){n}" for n in names) + "};\n"
        "  printf(\"%zu %d\\n\", sizeof(fns) / sizeof(fns[0]), pa_abi_version());\n"
        "  printf(\"%zu\\n\", sizeof(pa_kv_desc));\n"
        + "".join(f"  printf(\"%zu\\n\", offsetof(pa_kv_desc, {f}));\n" for f in fields) +
        "  return 0;\n}\n")
    exe = tmp_path / "caller"
    lib_dir = os.path.dirname(B.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                    "-o", str(exe), "-L", lib_dir, "-l:" + os.path.basename(B.LIB_PATH),
                    "-Wl,-rpath," + lib_dir], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == len(names) and int(out[1]) == B.ABI_VERSION
    assert int(out[2]) == ctypes.sizeof(B.PaKvDesc)
    assert [int(x) for x in out[3:]] == [getattr(B.PaKvDesc, f).offset for f in fields]
