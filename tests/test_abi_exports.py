"""CPU checks of the C-ABI library: it builds for sm_103a, loads without a
GPU and exports every function include/*.h declares; the host-only rollback
bookkeeping (gdn_commit) runs without a device."""
import ctypes as C
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from speculative_decode_verification_gb300 import binding, build

    build.build()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"verify_init", "q4_qmv_k", "q4_gather_experts_k", "gdn_verify_k", "gdn_commit"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_commit_bookkeeping_on_host(lib):
    from speculative_decode_verification_gb300 import binding as B

    st = B.GdnState()
    st.n_slots, st.cur, st.pending_k = 10, 3, 0
    assert lib.gdn_commit(C.byref(st), 0) == B.EINVAL  # nothing pending
    st.pending_k = 4
    for r, s in enumerate([3, 0, 1, 2, 4]):
        st.pending[r] = s
    assert lib.gdn_commit(C.byref(st), 5) == B.EINVAL  # beyond the verified rows
    assert lib.gdn_commit(C.byref(st), -1) == B.EINVAL
    assert lib.gdn_commit(C.byref(st), 2) == B.OK
    assert st.cur == 1 and st.pending_k == 0
    assert lib.gdn_commit(C.byref(st), 1) == B.EINVAL  # a second commit
    st.pending_k = 4
    assert lib.gdn_commit(C.byref(st), 0) == B.OK
    assert st.cur == 3


def test_null_context_is_rejected(lib):
    assert lib.q4_qmv_k(None, None, None, 1, None, 0, None) == 1
    assert lib.verify_last_error(None) == b"null context"


def test_attention_cache_bookkeeping_on_host(lib):
    from speculative_decode_verification_gb300 import binding as B

    c = B.KvCache()
    c.capacity, c.len, c.split, c.pending_k = 100, 10, 32, 0
    assert lib.attn_commit(C.byref(c), 0) == B.EINVAL  # nothing pending
    c.pending_k = 4
    assert lib.attn_commit(C.byref(c), 5) == B.EINVAL
    assert lib.attn_commit(C.byref(c), 3) == B.OK
    assert c.len == 13 and c.pending_k == 0
    p = B.attn_params(24, 2, 256)
    # rotated queries (hi, lo: per KV head 12 pairs in 128 rows), then (max,
    # sum) and outputs of 2 heads x 4 splits x 16 pairs
    want = 2 * (2 * 128 * 256 * 2) + 2 * 4 * 16 * 8 + 2 * 4 * 16 * 256 * 4
    assert B.attn_workspace_bytes(p, 1024, 256, 1) == want
    assert B.attn_workspace_bytes(p, 1024, 250, 1) == 0  # split not a multiple of 32
    assert B.attn_workspace_bytes(B.attn_params(24, 5, 256), 1024, 256, 1) == 0
    # default split: about 74 splits per KV head, a multiple of 64, at least 128
    assert B.attn_default_split(100) == 128 and B.attn_default_split(4128) == 128
    assert B.attn_default_split(65568) == 896 and -(-65568 // 896) == 74
