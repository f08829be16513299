"""The C-ABI library without a GPU: it loads, exports every entry point declared in
include/msa.h, and rejects invalid arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import block_sparse_attention_msa_gb300 as msa
from block_sparse_attention_msa_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_msa_gb300 import build
    build.build()
    return msa.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "msa.h")).read()
    return sorted(set(re.findall(r"^MSA_API [\w\s\*]*?\b(msa_\w+)\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("msa_index_score_topk", "msa_sparse_prefill", "msa_build_sparse_page_table",
                     "msa_paged_sparse_decode"):
        assert required in names
    assert sorted(n for n, _, _ in _lib.SIGNATURES) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.msa_version().decode() == "0.1.0"


def test_workspace_sizes(lib):
    assert lib.msa_index_score_topk_workspace_size(8, 1, 8, 469) >= 8 * 8 * 469 * 4 + 8 * 4
    assert lib.msa_index_score_topk_workspace_size(0, 1, 8, 469) == 0
    assert lib.msa_paged_sparse_decode_workspace_size(64, 64, 8, 16) >= 64 * 64 * 4 * 128 * 4
    assert lib.msa_sparse_prefill_workspace_size(32768, 32768, 64, 8, 16) > 32768 * 8 * 16 * 8 * 128 * 2
    assert lib.msa_prefill_bucket_workspace_size(1000, 8, 16, 256) >= 8 * 256 * 4 + 1000 * 8 * 16 * 4


def _err(lib):
    return lib.msa_last_error().decode()


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails host validation


def test_argument_validation_rejects_before_launch(lib):
    ws = ctypes.c_void_p(0x10000)
    # null pointer
    rc = lib.msa_index_score_topk(None, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 16, FAKE, None, ws,
                                  1 << 20, None)
    assert rc == -1 and "null" in _err(lib)
    # unsupported topk, Hkv, Di
    assert lib.msa_index_score_topk(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 65, FAKE, None, ws,
                                    1 << 20, None) == -3
    assert lib.msa_index_score_topk(FAKE, FAKE, FAKE, FAKE, 1, 1, 3, 128, 4, 4, 16, FAKE, None, ws,
                                    1 << 20, None) == -3
    assert lib.msa_index_score_topk(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 96, 4, 4, 16, FAKE, None, ws,
                                    1 << 20, None) == -3
    # workspace too small / misaligned
    assert lib.msa_index_score_topk(FAKE, FAKE, FAKE, FAKE, 8, 1, 8, 128, 469, 3752, 16, FAKE, None,
                                    ws, 16, None) == -4
    assert lib.msa_index_score_topk(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 16, FAKE, None,
                                    ctypes.c_void_p(0x10010), 1 << 20, None) == -4
    # N beyond the table
    assert lib.msa_index_score_topk(FAKE, FAKE, FAKE, FAKE, 1, 600, 8, 128, 4, 4, 16, FAKE, None, ws,
                                    1 << 30, None) == -2
    # decode: D != 128, bad GQA ratio, page-id overflow
    assert lib.msa_paged_sparse_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 64, 16, 10, FAKE,
                                       None, ws, 1 << 30, None) == -3
    assert lib.msa_paged_sparse_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 60, 8, 128, 16, 10, FAKE,
                                       None, ws, 1 << 30, None) == -3
    assert lib.msa_paged_sparse_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 128, 16, 1 << 22,
                                       FAKE, None, ws, 1 << 30, None) == -3
    # prefill: T > S_kv, D
    assert lib.msa_sparse_prefill(FAKE, FAKE, FAKE, FAKE, 100, 50, 64, 8, 128, 16, FAKE, None, ws,
                                  1 << 30, None) == -1
    assert lib.msa_sparse_prefill(FAKE, FAKE, FAKE, FAKE, 100, 200, 64, 8, 256, 16, FAKE, None, ws,
                                  1 << 30, None) == -3
    # paged prefill: null page table, bad page count, then the shared checks
    assert lib.msa_sparse_prefill_paged(FAKE, FAKE, FAKE, None, 16, FAKE, 100, 200, 64, 8, 128, 16,
                                        FAKE, None, ws, 1 << 30, None) == -1
    assert lib.msa_sparse_prefill_paged(FAKE, FAKE, FAKE, FAKE, 0, FAKE, 100, 200, 64, 8, 128, 16,
                                        FAKE, None, ws, 1 << 30, None) == -1
    assert lib.msa_sparse_prefill_paged(FAKE, FAKE, FAKE, FAKE, 16, FAKE, 100, 200, 64, 8, 256, 16,
                                        FAKE, None, ws, 1 << 30, None) == -3
    # KV staging: null stage output, D
    assert lib.msa_stage_selected_kv(FAKE, FAKE, 16, FAKE, 4, 8, 128, 16, FAKE, None, FAKE,
                                     None) == -1
    assert lib.msa_stage_selected_kv(FAKE, FAKE, 16, FAKE, 4, 8, 64, 16, FAKE, FAKE, FAKE,
                                     None) == -3
    # page table: null output
    assert lib.msa_build_sparse_page_table(FAKE, FAKE, FAKE, 1, 1, 8, 16, 4, 4, None, FAKE,
                                           None) == -1
    # merge: bad sizes
    assert lib.msa_lse_merge(FAKE, 1, FAKE, 4, 0, 8, 128, FAKE, None, None) == -1
    # empty inputs are a no-op success
    assert lib.msa_index_score_topk(None, None, None, None, 0, 1, 8, 128, 4, 4, 16, None, None,
                                    None, 0, None) == 0
    assert lib.msa_sparse_prefill(None, None, None, None, 0, 0, 64, 8, 128, 16, None, None, None,
                                  0, None) == 0


def test_fused_scratch_and_bucket_entry_points_reject_before_launch(lib):
    ws = ctypes.c_void_p(0x10000)
    # scorer + page table: a null page-table output, then the scorer's own checks
    assert lib.msa_index_score_topk_page_table(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 16,
                                               FAKE, None, None, FAKE, ws, 1 << 20, None) == -1
    assert "page-table output" in _err(lib)
    assert lib.msa_index_score_topk_page_table(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 96, 4, 4, 16,
                                               FAKE, None, FAKE, FAKE, ws, 1 << 20, None) == -3
    assert lib.msa_index_score_topk_page_table(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 16,
                                               FAKE, None, FAKE, FAKE, ws, 16, None) == -4
    # scorer without a workspace: the same argument errors as the workspace entry point, found
    # before the call looks for its device scratch (no device here)
    assert lib.msa_index_score_topk_noalloc(None, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 16,
                                            FAKE, None, None) == -1
    assert "null" in _err(lib) and "noalloc" in _err(lib)
    assert lib.msa_index_score_topk_noalloc(FAKE, FAKE, FAKE, FAKE, 1, 1, 8, 128, 4, 4, 65,
                                            FAKE, None, None) == -3
    assert lib.msa_index_score_topk_noalloc(FAKE, FAKE, FAKE, FAKE, 1, 600, 8, 128, 4, 4, 16,
                                            FAKE, None, None) == -2
    # ... and calls whose block scores exceed the 8 MiB scratch, before any device work
    assert lib.msa_index_score_topk_noalloc(FAKE, FAKE, FAKE, FAKE, 64, 1, 8, 128, 8192, 1, 16,
                                            FAKE, None, None) == -3
    assert "scratch" in _err(lib)
    assert lib.msa_index_score_topk_noalloc(None, None, None, None, 0, 1, 8, 128, 4, 4, 16,
                                            None, None, None) == 0
    # bucketing: null output, group count, list sizes beyond int32, workspace
    assert lib.msa_prefill_bucket(FAKE, 100, 8, 16, 4, None, FAKE, ws, 1 << 20, None) == -1
    assert lib.msa_prefill_bucket(FAKE, 100, 17, 16, 4, FAKE, FAKE, ws, 1 << 20, None) == -1
    assert lib.msa_prefill_bucket(FAKE, 1 << 30, 8, 16, 4, FAKE, FAKE, ws, 1 << 20, None) == -3
    assert lib.msa_prefill_bucket(FAKE, 100, 8, 16, 4, FAKE, FAKE, ws, 16, None) == -4
    assert lib.msa_prefill_bucket(FAKE, 100, 8, 16, 4, FAKE, FAKE, ctypes.c_void_p(0x10010),
                                  1 << 20, None) == -4


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError, match="CUDA"):
        msa.sparse_prefill(torch.zeros(1, 8, 128, dtype=torch.bfloat16),
                           torch.zeros(1, 1, 128, dtype=torch.bfloat16),
                           torch.zeros(1, 1, 128, dtype=torch.bfloat16),
                           torch.zeros(1, 1, 2, dtype=torch.int32))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no CPU fallback: without the built library every call path stops at load()
    from block_sparse_attention_msa_gb300 import build as _build
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "libmsa_gb300.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        msa.load()


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "msa.h"

int main(void) {
  /* a C caller sees the library only through msa.h */
  if (strcmp(msa_version(), "0.1.0") != 0) return 1;
  size_t need = msa_index_score_topk_workspace_size(8, 1, 8, 469);
  if (need < (size_t)8 * 8 * 469 * 4) return 2;
  /* host checks run before any device call: a null q_idx is MSA_ERR_ARG */
  int32_t ids[16];
  int rc = msa_index_score_topk(NULL, NULL, NULL, NULL, 1, 1, 8, 128, 4, 4, 16, ids, NULL,
                                NULL, 0, NULL);
  if (rc != MSA_ERR_ARG || strstr(msa_last_error(), "null") == NULL) return 3;
  printf("ok\n");
  return 0;
}
"""


def test_header_compiles_as_c_and_links_the_library(lib, tmp_path):
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    so = msa.library_path()
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(exe), so,
                    "-Wl,-rpath," + os.path.dirname(so)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
