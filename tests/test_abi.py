"""The C-ABI library builds for sm_103a, loads, and exports every function
that include/pa.h declares (no compute calls: runs without a GPU)."""
import ctypes
import glob
import os
import re

from paged_kv_cache_143_gb300 import pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pa_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(pa.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(pa.lib()._name)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_host_side_rejections():
    L = pa.lib()
    assert pa.status_string(pa.PA_OK) == "PA_OK"
    for s in range(6):
        assert pa.status_string(s)
    # argument errors are found on the host before any CUDA call
    assert L.pa_write_kv(None, None, None, None, 1, None) == pa.PA_ERR_INVALID
    assert L.pa_copy_blocks(None, None, None, 1, None) == pa.PA_ERR_INVALID
    assert L.pa_apply_staged_writes(None, 1, 1, None, None, None, None, -1, None, 0, None,
                                    None) == pa.PA_ERR_INVALID
    pool = pa._Pool(16, 16, 4, 16, 1, 64, 0, 1.0, 1.0)
    assert L.pa_write_kv(ctypes.byref(pool), None, None, None, 0, None) == pa.PA_OK
    bad = pa._Pool(16, 16, 4, 24, 1, 64, 0, 1.0, 1.0)  # block size 24
    assert L.pa_write_kv(ctypes.byref(bad), None, None, None, 0, None) == pa.PA_ERR_UNSUPPORTED
    bad = pa._Pool(16, 16, 4, 16, 1, 96, 0, 1.0, 1.0)  # head dim 96
    assert L.pa_copy_blocks(ctypes.byref(bad), None, None, 0, None) == pa.PA_ERR_UNSUPPORTED
    fp8 = pa._Pool(16, 16, 4, 16, 1, 64, 1, 0.0, 1.0)  # FP8 with zero scale
    assert L.pa_write_kv(ctypes.byref(fp8), None, None, None, 0, None) == pa.PA_ERR_INVALID
    mis = pa._Pool(17, 16, 4, 16, 1, 64, 0, 1.0, 1.0)  # misaligned pool
    assert L.pa_write_kv(ctypes.byref(mis), None, None, None, 0, None) == pa.PA_ERR_INVALID
    # a pool of no blocks cannot hold any request's keys (fake, aligned device
    # pointers: the call returns before touching them)
    import numpy as np
    empty = pa._Pool(16, 16, 0, 16, 1, 64, 0, 1.0, 1.0)
    qsl, seq = np.array([0, 1], np.int32), np.array([5], np.int32)
    assert L.pa_forward(16, 16, 16, 16, qsl.ctypes.data_as(ctypes.c_void_p),
                        seq.ctypes.data_as(ctypes.c_void_p), 16, 1, 1, 1, 1,
                        ctypes.byref(empty), 0.125, 1, None, 0, None) == pa.PA_ERR_INVALID


def test_workspace_size_formula():
    # the plan area of the persistent decode (R + 3 int32 words, rounded up to
    # 256 bytes), then per split slot an fp32 partial row and its (max, sum)
    plan = (4 * (256 + 3) + 255) // 256 * 256
    assert pa.forward_workspace_size(256, 32, 128, 4) == plan + 256 * 32 * 4 * (128 * 4 + 8)
    assert pa.forward_workspace_size(1, 1, 64, 1) == 256 + (64 * 4 + 8)
    assert pa.forward_workspace_size(0, 32, 128, 4) == 0


def test_shared_prefix_host_rejections():
    """Group arguments of pa_forward_shared_prefix are checked on the host
    before any CUDA call (fake, aligned device pointers are never touched)."""
    import numpy as np
    L = pa.lib()
    pool = pa._Pool(16, 16, 32, 16, 4, 64, 0, 1.0, 1.0)
    i32 = lambda *v: np.array(v, np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)

    def call(qsl, seq, first, size, prefix, G=None, ws_bytes=1 << 20):
        G = len(first) if G is None else G
        R = len(seq)
        return L.pa_forward_shared_prefix(
            16, 16, 16, 16, ptr(qsl), ptr(seq), 16, 4, R, int(qsl[-1]), 4, ctypes.byref(pool),
            0.125, 1, G, ptr(first), ptr(size), ptr(prefix), 16 if ws_bytes else None, ws_bytes,
            None)

    qsl, seq = i32(0, 1, 2, 3), i32(40, 50, 60)
    assert call(qsl, seq, i32(0), i32(2), i32(2), G=65) == pa.PA_ERR_UNSUPPORTED
    assert call(qsl, seq, i32(0), i32(2), i32(3)) == pa.PA_ERR_INVALID  # seq 40 <= prefix 48
    assert call(qsl, seq, i32(0), i32(2), i32(0)) == pa.PA_ERR_INVALID  # empty prefix
    assert call(qsl, seq, i32(0), i32(2), i32(5)) == pa.PA_ERR_INVALID  # prefix > max_blocks
    assert call(qsl, seq, i32(0), i32(0), i32(2)) == pa.PA_ERR_INVALID  # empty group
    assert call(qsl, seq, i32(2), i32(2), i32(2)) == pa.PA_ERR_INVALID  # past num_reqs
    assert call(qsl, seq, i32(0, 1), i32(2, 2), i32(2, 2)) == pa.PA_ERR_INVALID  # overlap
    assert call(qsl, seq, i32(1, 0), i32(1, 1), i32(2, 2)) == pa.PA_ERR_INVALID  # unordered
    assert call(qsl, seq, i32(-1), i32(2), i32(2)) == pa.PA_ERR_INVALID
    assert call(i32(0, 1, 2, 5), seq, i32(1), i32(2), i32(1)) == pa.PA_ERR_INVALID  # a prefill
    # one prefix piece and one tail split per request do not fit in no workspace
    assert call(qsl, seq, i32(0), i32(2), i32(2), ws_bytes=0) == pa.PA_ERR_INVALID
    one_split = pa.forward_workspace_size(3, 4, 64, 1)
    assert call(qsl, seq, i32(0), i32(2), i32(2), ws_bytes=one_split) == pa.PA_ERR_INVALID


C_PROGRAM = r"""
#include <stdio.h>
#include "pa.h"
#include "pa_sched.h"

static const void* const every_entry_point[] = {
%s
};

int main(void) {
  size_t i, n = sizeof every_entry_point / sizeof every_entry_point[0];
  for (i = 0; i < n; ++i)
    if (!every_entry_point[i]) return 2;
  pa_sched_config cfg = {64, 16, 8, 16, 256, 128, 1};
  pa_sched* s = NULL;
  if (pa_sched_create(&cfg, &s) != PA_OK) return 3;
  int32_t prompt[40];
  for (i = 0; i < 40; ++i) prompt[i] = (int32_t)i;
  if (pa_sched_add_request(s, 7, prompt, 40, 2, 0) != PA_OK) return 4;
  pa_sched_batch b;
  if (pa_sched_step(s, &b) != PA_OK) return 5;
  printf("%%d %%d %%d %%lld\n", b.num_reqs, b.num_tokens, b.num_decode, (long long)b.req_ids[0]);
  int32_t sampled[1] = {99}, num_finished = 0;
  if (pa_sched_commit(s, sampled, b.num_reqs, NULL, 0, &num_finished) != PA_OK) return 6;
  if (pa_sched_step(s, &b) != PA_OK) return 7;
  printf("%%d %%d %%d %%d\n", b.num_reqs, b.num_tokens, b.num_decode, b.positions[0]);
  printf("%%s\n", pa_status_string(PA_ERR_INVALID));
  pa_sched_destroy(s);
  return 0;
}
"""


def _compile_and_link(tmp_path, compiler, flags, suffix):
    import shutil
    import subprocess
    if shutil.which(compiler) is None:
        import pytest
        pytest.skip(f"{compiler} not available")
    lib_dir = os.path.dirname(pa.lib()._name)
    src = tmp_path / f"use_pa.{suffix}"
    refs = ",\n".join(f"    (const void*)&{name}" for name in declared_functions())
    src.write_text(C_PROGRAM % refs)
    exe = tmp_path / f"use_pa_{suffix}"
    r = subprocess.run([compiler, *flags, "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", lib_dir, "-lpa", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_headers_build_a_plain_c_program_that_drives_the_scheduler(tmp_path):
    """Both headers compile as C99 and as C++17 against the library, every
    declared entry point links, and the host-only scheduler runs from C:
    a 40-token prompt is one 40-token chunk, then one decode at position 40."""
    import subprocess
    exe = _compile_and_link(tmp_path, "gcc", ["-std=c99"], "c")
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    lines = r.stdout.splitlines()
    assert lines[0] == "1 40 0 7"
    assert lines[1] == "1 1 1 40"
    assert lines[2] == pa.status_string(pa.PA_ERR_INVALID)
    _compile_and_link(tmp_path, "g++", ["-std=c++17"], "cpp")


def test_pool_struct_is_cached_and_rebuilt_on_reassignment(monkeypatch):
    """KVPool.ref() hands the C ABI one struct per pool; reassigning a scale
    or a tensor rebuilds it (CPU tensors stand in for device ones: only
    their addresses are read)."""
    import torch
    monkeypatch.setattr(pa, "_dptr", lambda t, dtype=None: t.data_ptr() if t.numel() else None)
    k = torch.zeros(8, 2, 16, 64, dtype=torch.uint8)
    v = torch.zeros_like(k)
    pool = pa.KVPool(k, v, 0.5, 0.25)
    read = lambda r: ctypes.cast(r, ctypes.POINTER(pa._Pool)).contents
    r = pool.ref()
    s = read(r)
    assert (s.k_pool, s.v_pool) == (k.data_ptr(), v.data_ptr())
    assert (s.num_blocks, s.num_kv_heads, s.block_size, s.head_dim) == (8, 2, 16, 64)
    assert (s.dtype, s.k_scale, s.v_scale) == (pa.PA_KV_FP8_E4M3, 0.5, 0.25)
    assert pool.ref() is r
    pool.k_scale = 2.0
    assert pool.ref() is not r and read(pool.ref()).k_scale == 2.0
    k2 = torch.zeros_like(k)
    pool.k = k2
    assert read(pool.ref()).k_pool == k2.data_ptr()
    # the storage moved under the same attribute (set_ swaps it in place)
    r2 = pool.ref()
    v2 = torch.zeros_like(v)
    pool.v.set_(v2)
    assert pool.ref() is not r2 and read(pool.ref()).v_pool == v2.data_ptr()


def test_prefill_gqa_wider_than_a_tile_is_refused():
    """A prefill tile holds 128 rows of token x head: a chunk whose GQA group
    is wider (g = Hq / Hkv > 128) is refused on the host, before any launch."""
    import numpy as np
    L = pa.lib()
    pool = pa._Pool(16, 16, 4, 16, 1, 64, pa.PA_KV_BF16, 1.0, 1.0)
    qsl = np.array([0, 3], np.int32)
    seq = np.array([8], np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = L.pa_forward(16, 16, 16, 16, ptr(qsl), ptr(seq), 16, 4, 1, 3, 256,
                      ctypes.byref(pool), 0.125, 1, None, 0, None)
    assert st == pa.PA_ERR_UNSUPPORTED


def test_gather_rows_host_rejections():
    """pa_gather_rows checks its arguments on the host before any launch
    (fake, aligned device pointers are never touched)."""
    L = pa.lib()
    assert L.pa_gather_rows(16, 10, 256, 16, 0, 16, None) == pa.PA_OK  # nothing to gather
    assert L.pa_gather_rows(16, 10, 256, 16, -1, 16, None) == pa.PA_ERR_INVALID
    assert L.pa_gather_rows(16, 10, 24, 16, 3, 16, None) == pa.PA_ERR_INVALID  # not 16-byte rows
    assert L.pa_gather_rows(16, 10, 0, 16, 3, 16, None) == pa.PA_ERR_INVALID
    assert L.pa_gather_rows(None, 10, 256, 16, 3, 16, None) == pa.PA_ERR_INVALID
    assert L.pa_gather_rows(16, 10, 256, None, 3, 16, None) == pa.PA_ERR_INVALID
    assert L.pa_gather_rows(24, 10, 256, 16, 3, 16, None) == pa.PA_ERR_INVALID  # misaligned src
    assert L.pa_gather_rows(16, -1, 256, 16, 3, 16, None) == pa.PA_ERR_INVALID
