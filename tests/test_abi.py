"""The C-ABI library loads and exports every entry point include/sv.h
declares; host-side argument validation rejects bad calls before any CUDA
work is enqueued (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "sv.h")).read()
    return sorted(set(re.findall(r"^SV_API\s+[\w\s\*]+?\b(sv_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_sv_gb300 import build
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_five_calls():
    names = _declared()
    for fn in ("sv_verify_attn", "sv_lm_head", "sv_accept_greedy", "sv_accept_sample", "sv_kv_commit"):
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 14
    for fn in names:
        assert hasattr(lib, fn), fn


def test_binding_imports_without_gpu():
    from speculative_decoding_verification_sv_gb300 import binding
    assert binding.lib.sv_version() == 100
    assert binding.lib.sv_status_string(3) == b"unsupported configuration"


def test_host_validation_rejects_before_launch(lib):
    from speculative_decoding_verification_sv_gb300 import binding as b
    L = b.lib
    P = ctypes.c_void_p
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: validation fails first
    # NULL pointers
    assert L.sv_lm_head(None, fake, fake, 5, 1536, 151936, None) == 1
    # misaligned pointer
    assert L.sv_lm_head(ctypes.c_void_p(0x10002), fake, fake, 5, 1536, 151936, None) == 1
    # bad shapes
    assert L.sv_lm_head(fake, fake, fake, 0, 1536, 151936, None) == 2
    assert L.sv_lm_head(fake, fake, fake, 5, 1537, 151936, None) == 2
    # head dim other than 128 is unsupported
    s = b._AttnShape(1, 5, 12, 2, 64, 4096)
    assert L.sv_verify_attn(ctypes.byref(s), fake, fake, fake, fake, fake, fake, None, ctypes.c_float(0.1), fake,
                            fake, 1 << 30, None) == 3
    s = b._AttnShape(1, 5, 12, 5, 128, 4096)   # Hq % Hkv != 0
    assert L.sv_verify_attn(ctypes.byref(s), fake, fake, fake, fake, fake, fake, None, ctypes.c_float(0.1), fake,
                            fake, 1 << 30, None) == 2
    # batch 1, 32K context: several clusters per KV head meet in the
    # workspace, which is then required (NULL -> argument error, short ->
    # workspace error); at 4K context one cluster per KV head needs none
    assert L.sv_verify_attn_workspace(ctypes.byref(b._AttnShape(1, 5, 12, 2, 128, 4224))) == 0
    s = b._AttnShape(1, 5, 12, 2, 128, 32832)
    need = L.sv_verify_attn_workspace(ctypes.byref(s))
    assert need > 0 and need % 16 == 0
    assert L.sv_verify_attn(ctypes.byref(s), fake, fake, fake, fake, fake, fake, None, ctypes.c_float(0.1), fake,
                            None, need, None) == 1
    assert L.sv_verify_attn(ctypes.byref(s), fake, fake, fake, fake, fake, fake, None, ctypes.c_float(0.1), fake,
                            fake, need - 16, None) == 4
    # launch flags: only SV_ATTN_CACHE_READY (1) is defined
    s = b._AttnShape(1, 5, 12, 2, 128, 4224)
    assert L.sv_verify_attn_ex(ctypes.byref(s), fake, fake, fake, fake, fake, fake, None, ctypes.c_float(0.1), fake,
                               None, 0, 2, None) == 1
    assert L.sv_verify_attn_ex(ctypes.byref(s), None, fake, fake, fake, fake, fake, None, ctypes.c_float(0.1), fake,
                               None, 0, 1, None) == 1
    assert L.sv_lm_head_ex(fake, fake, fake, 5, 1536, 151936, 2, None) == 1
    assert L.sv_lm_head_ex(None, fake, fake, 5, 1536, 151936, 1, None) == 1
    # short workspace
    assert L.sv_accept_greedy(fake, fake, None, 1, 5, 151936, fake, fake, fake, fake, 8, None) == 4
    # temperature must be positive; vocab must be a multiple of 4
    args = [fake, fake, 151936, fake, None, 64, 9, 151936, ctypes.c_float(0.0), 1, 0, None, fake, fake, fake, fake,
            1 << 20, None]
    assert L.sv_accept_sample(*args) == 1
    args[8] = ctypes.c_float(1.0)
    args[7] = 151937
    assert L.sv_accept_sample(*args) == 2
    # commit: R above 128
    assert L.sv_kv_commit(fake, fake, fake, fake, 28, 1, 2, 128, 4224, 200, fake, fake, fake, None) == 2
    # paged attention: T_cap must be max_pages * 64; a page table is required
    s = b._AttnShape(1, 5, 12, 2, 128, 4224)
    assert L.sv_verify_attn_paged(ctypes.byref(s), fake, fake, fake, 100, fake, 65, fake, fake, fake, None,
                                  ctypes.c_float(0.1), fake, fake, 1 << 30, 0, None) == 2
    assert L.sv_verify_attn_paged(ctypes.byref(s), fake, fake, fake, 100, None, 66, fake, fake, fake, None,
                                  ctypes.c_float(0.1), fake, fake, 1 << 30, 0, None) == 1
    assert L.sv_kv_commit_paged(fake, fake, 0, fake, 4, fake, fake, 28, 1, 2, 128, 5, fake, fake, fake, None) == 2
    assert L.sv_kv_commit_paged(fake, fake, 8, None, 4, fake, fake, 28, 1, 2, 128, 5, fake, fake, fake, None) == 1
    # relaxed acceptance: delta must be >= 0 and not NaN; short workspace
    for bad in (-0.5, float("nan")):
        assert L.sv_accept_greedy_relaxed(fake, fake, None, 1, 5, 151936, ctypes.c_float(bad), fake, fake, fake,
                                          fake, 1 << 20, None) == 1
    assert L.sv_accept_greedy_relaxed(fake, fake, None, 1, 5, 151936, ctypes.c_float(1.0), fake, fake, fake, fake,
                                      8, None) == 4
    # LM head with argmax keys: the key buffer is required and sized by the query;
    # unknown flags rejected; logits may be NULL
    need = L.sv_lm_head_argmax_bytes(5, 151936)
    assert need == 5 * 1187 * 8
    assert L.sv_lm_head_argmax(fake, fake, None, 5, 1536, 151936, None, need, 0, None) == 1
    assert L.sv_lm_head_argmax(fake, fake, None, 5, 1536, 151936, fake, need - 8, 0, None) == 4
    assert L.sv_lm_head_argmax(fake, fake, None, 5, 1536, 151936, fake, need, 2, None) == 1
    assert L.sv_lm_head_argmax(fake, fake, None, 5, 1537, 151936, fake, need, 0, None) == 2
    # fused acceptance + commit: a commit needs all four cache buffers; R <= 128
    assert L.sv_accept_greedy_commit(fake, fake, None, 1, 5, 151936, fake, fake, fake, None, fake, None, None, 28, 2,
                                     128, 4224, fake, None) == 1
    assert L.sv_accept_greedy_commit(fake, fake, None, 1, 200, 151936, fake, fake, fake, None, None, None, None, 0, 0,
                                     0, 0, None, None) == 2
    assert L.sv_accept_greedy_commit(None, fake, None, 1, 5, 151936, fake, fake, fake, None, None, None, None, 0, 0,
                                     0, 0, None, None) == 1
    assert L.sv_accept_greedy_commit_paged(fake, fake, None, 1, 5, 151936, fake, fake, fake, fake, fake, 0, fake, 4,
                                           fake, fake, 28, 2, 128, fake, None) == 2
    assert L.sv_accept_greedy_commit_paged(fake, fake, None, 1, 5, 151936, fake, fake, fake, fake, fake, 8, None, 4,
                                           fake, fake, 28, 2, 128, fake, None) == 1


def test_copy_host_validation(lib):
    """sv_copy: nothing to do is OK; NULLs, overlapping ranges and pageable
    host memory are refused before any launch."""
    from speculative_decoding_verification_sv_gb300 import binding as b
    L = b.lib
    fake = ctypes.c_void_p(0x10000)
    assert L.sv_copy(None, None, 0, None) == 0
    assert L.sv_copy(None, fake, 16, None) == 1
    assert L.sv_copy(fake, None, 16, None) == 1
    buf = ctypes.create_string_buffer(64)   # pageable host memory
    base = ctypes.addressof(buf)
    assert L.sv_copy(ctypes.c_void_p(base + 32), ctypes.c_void_p(base), 16, None) == 1
    assert L.sv_copy(ctypes.c_void_p(base + 8), ctypes.c_void_p(base), 16, None) == 1   # overlapping


def test_workspace_queries(lib):
    from speculative_decoding_verification_sv_gb300 import binding as b
    assert b.lib.sv_accept_greedy_workspace(16, 9, 152064) == 16 * 9 * 19 * 8
    # row statistics, then the chain path's per-sequence records and sums
    assert b.lib.sv_accept_sample_workspace(64, 9, 151936) == 64 * 9 * 8 + 64 * 16 + 64 * 2 * (64 * 32 + 64) * 4
    # 7B batch 16: 63 rows per (sequence, KV head) in 64-row tiles, one cluster
    # each, merged on chip
    assert b.verify_attn_workspace(16, 9, 28, 4, 128, 8320) == 0


def test_sample_shapes_checked(lib):
    """The binding refuses a q whose row count does not match the mode (R - 1
    rows for a chain, R for a tree): the C ABI cannot see it."""
    import torch
    from speculative_decoding_verification_sv_gb300 import binding as b
    lg = torch.zeros(1, 5, 16)
    tok = torch.zeros(1, 5, dtype=torch.int32)
    par = torch.tensor([[-1, 0, 0, 1, 1]], dtype=torch.int32)
    with pytest.raises(ValueError):
        b.accept_sample(lg, torch.zeros(1, 5, 16), tok)          # a chain wants 4 rows of q
    with pytest.raises(ValueError):
        b.accept_sample(lg, torch.zeros(1, 4, 16), tok, par)     # a tree wants 5
    with pytest.raises(ValueError):
        b.accept_sample_noalloc(lg, torch.zeros(1, 4, 16), tok, par)
