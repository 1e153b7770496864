"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol declared in include/*.h, sizes workspaces, and rejects bad arguments
before enqueueing anything."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# Every test runs twice: once in the CPU tier and once, unchanged, in the GPU
# tier, so the host-side contract is also checked on the machine that runs the
# kernels (the library must load and validate identically with a driver present).
@pytest.fixture(scope="module", params=[pytest.param("host"),
                                        pytest.param("gpu-box", marks=pytest.mark.gpu)])
def lib(request):
    from block_sparse_attention_nsa_gb300 import build
    build.build()
    import block_sparse_attention_nsa_gb300 as nsa
    return nsa.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"NSA_API\s+[\w\s\*]+?\b(nsa_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert len(declared) >= 10
    so = os.path.join(ROOT, "block_sparse_attention_nsa_gb300", "libnsa_sel.so")
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (nsa_\w+)", out))
    assert declared <= exported, declared - exported
    for name in declared:
        assert getattr(lib, name) is not None


def _dims(**kw):
    import block_sparse_attention_nsa_gb300 as nsa
    base = dict(num_seqs=1, total_tokens=8192, h_q=4, h_k=4, head_dim=128, block_size=64,
                topk=16, dtype=0)
    base.update(kw)
    return nsa.Dims(**base)


def test_workspace_size_and_envelope(lib):
    import block_sparse_attention_nsa_gb300 as nsa
    f, b = nsa.workspace_size(_dims())
    assert f > 0 and b > 0
    # compact partial buffer bound: h_k * N * T rows of d 16-bit values
    assert f >= 4 * 8192 * 16 * 128 * 2
    bad = [dict(head_dim=96), dict(block_size=48), dict(topk=33), dict(dtype=7), dict(h_q=6),
           dict(h_k=0), dict(num_seqs=0), dict(total_tokens=-1)]
    for kw in bad:
        with pytest.raises(nsa.NsaError):
            nsa.workspace_size(_dims(**kw))
    # too many pairs for 32-bit positions
    with pytest.raises(nsa.NsaError) as e:
        nsa.workspace_size(_dims(total_tokens=1 << 27, topk=32))
    assert e.value.code == 2


def test_validation_returns_before_launch(lib):
    d = _dims()
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: every call below fails validation
    st = lib.nsa_sel_attn_fwd(ctypes.byref(d), fake, fake, fake, fake, fake, 0.1, fake, fake,
                              fake, 16, None)
    assert st == 3                       # workspace too small
    st = lib.nsa_sel_attn_fwd(ctypes.byref(d), None, fake, fake, fake, fake, 0.1, fake, fake,
                              fake, 1 << 40, None)
    assert st == 1                       # null q
    odd = ctypes.c_void_p((1 << 20) + 8)
    st = lib.nsa_sel_attn_fwd(ctypes.byref(d), odd, fake, fake, fake, fake, 0.1, fake, fake,
                              fake, 1 << 40, None)
    assert st == 1                       # q not 16-byte aligned
    st = lib.nsa_sel_attn_fwd(ctypes.byref(d), fake, fake, fake, fake, fake, float("nan"), fake,
                              fake, fake, 1 << 40, None)
    assert st == 1                       # non-finite scale
    d256 = _dims(head_dim=256, block_size=128)
    st = lib.nsa_sel_attn_bwd(ctypes.byref(d256), fake, fake, fake, fake, fake, 0.1, fake, fake,
                              fake, fake, fake, fake, fake, 1 << 40, 0, None)
    assert st == 2                       # backward with d = 256 needs B_K <= 64
    st = lib.nsa_sel_attn_index(None, fake, fake, fake, 1 << 40, None)
    assert st == 1
    d128 = _dims(head_dim=128, block_size=128)   # attention kernels not offered for this pair
    st = lib.nsa_sel_attn_fwd(ctypes.byref(d128), fake, fake, fake, fake, fake, 0.1, fake, fake,
                              fake, 1 << 40, None)
    assert st == 2


def test_compressed_branch_validation_returns_before_launch(lib):
    # nsa_compress_kv / nsa_cmp_attn_select reject bad arguments before any launch
    d = _dims()
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 8)
    st = lib.nsa_compress_kv(ctypes.byref(d), fake, 16, 32, fake, fake, fake, fake, fake, None,
                             None)
    assert st == 1                       # kernel_size < kernel_stride
    st = lib.nsa_compress_kv(ctypes.byref(d), fake, 32, 16, odd, fake, fake, fake, fake, None,
                             None)
    assert st == 1                       # k not 16-byte aligned
    st = lib.nsa_compress_kv(ctypes.byref(_dims(head_dim=256)), fake, 32, 16, fake, fake, fake,
                             fake, fake, None, None)
    assert st == 2                       # d = 256 not offered
    args = (fake, fake, fake, fake, fake, 32, 16)
    st = lib.nsa_cmp_attn_select(ctypes.byref(d), *args, 0, 0.1, 1, 2, fake, fake, fake, None,
                                 None, 0, None)
    assert st == 1                       # max_seqlen < 1
    st = lib.nsa_cmp_attn_select(ctypes.byref(d), *args, 8192, 0.1, -1, 2, fake, fake, fake,
                                 None, None, 0, None)
    assert st == 1                       # negative init_blocks
    st = lib.nsa_cmp_attn_select(ctypes.byref(d), *args, 1 << 30, 0.1, 1, 2, fake, fake, fake,
                                 None, None, 0, None)
    assert st == 2                       # importance rows beyond any supported length
    # one 64K sequence at g = 1: the rows leave a shared-memory CTA two warps, so a
    # workspace holding them for 128-token CTAs is asked for, and a short one refused
    d1 = _dims(h_q=d.h_k)
    b = ctypes.c_size_t()
    assert lib.nsa_cmp_workspace_size(ctypes.byref(d1), 32, 16, 65536, ctypes.byref(b)) == 0
    ctas = -(-d1.total_tokens // 128) * d1.h_k
    assert b.value == ctas * 128 * 1024 * 4
    st = lib.nsa_cmp_attn_select(ctypes.byref(d1), *args, 65536, 0.1, 1, 2, fake, fake, fake,
                                 None, fake, 16, None)
    assert st == 3                       # workspace too small
    assert lib.nsa_cmp_workspace_size(ctypes.byref(d1), 32, 16, 4096, ctypes.byref(b)) == 0
    assert b.value == 0                  # short sequences: shared memory suffices


def test_status_strings_and_kernel_names(lib):
    import block_sparse_attention_nsa_gb300 as nsa
    for code in range(7):
        assert lib.nsa_status_string(code)
    names = nsa.kernel_names()
    assert "fwd_main" in names and "index_scatter" in names and "bwd_main" in names
