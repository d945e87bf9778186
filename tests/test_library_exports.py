"""The C-ABI library builds, loads and exports every symbol include/attnres.h
declares; its host-only logic (source counts, source lists, argument and
order checks) behaves as specified.  No compute call: runs without a GPU."""
import ctypes
import os
import re

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    import __graft_entry__
    B = __graft_entry__._build_module()
    if not os.path.exists(B.LIB_PATH):
        B.build()
    from depth_wise_attention_block_gb300 import _native
    return _native


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "attnres.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attnres_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(native):
    declared = _declared_functions()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(native.lib, name), name
    assert sorted(native.EXPORTED) == declared


def test_abi_version_and_status_strings(native):
    v = native.lib.attnres_version()
    assert v >> 16 == 2
    for code in [0, -1, -2, -4, -5, -6]:
        assert native.lib.attnres_status_string(code).startswith(b"ATTNRES_")
    assert b"unknown" in native.lib.attnres_status_string(12345)


@pytest.mark.parametrize("L,B", [(93, 12), (7, 3), (6, 1), (5, 5), (5, 9), (1, 1), (13, 4)])
def test_num_sources_matches_the_value_list(native, L, B):
    for l in range(1, L + 2):
        assert native.lib.attnres_num_sources(l, B, L) == O.num_sources(l, B, L)
    assert native.lib.attnres_num_sources(L + 1, B, L) == -(-L // B) + 1
    assert native.lib.attnres_num_sources(0, B, L) == native.ATTNRES_EINVAL
    assert native.lib.attnres_num_sources(L + 2, B, L) == native.ATTNRES_EINVAL
    assert native.lib.attnres_num_sources(1, 0, L) == native.ATTNRES_EINVAL


def _fake_state(native, L, B, T=4, d=8, dtype=1):
    """State over fake (never dereferenced) device pointers."""
    N = -(-L // B)
    st = native.AttnresState()
    st.flags = 0x7F   # init clears the flags
    h0, partial = 0x10000, 0x20000
    reps = (ctypes.c_void_p * N)(*[0x100000 * (k + 1) for k in range(N)])
    rc = native.lib.attnres_state_init(ctypes.byref(st), h0, reps, N, partial, T, d, dtype, L, B, 1e-5)
    assert rc == 0, native.lib.attnres_last_error()
    assert st.flags == 0
    return st, h0, partial, list(reps)


@pytest.mark.parametrize("L,B", [(93, 12), (7, 3), (6, 1), (5, 9)])
def test_layer_sources_follow_eq10(native, L, B):
    st, h0, partial, reps = _fake_state(native, L, B)
    assert st.T == 4 and st.d == 8 and st.dtype == 1 and st.num_layers == L and st.block_size == B
    assert abs(st.eps - 1e-5) < 1e-12 and st.folded == 0
    out = (ctypes.c_void_p * 128)()
    n = ctypes.c_int()
    for l in range(1, L + 2):
        st.folded = l - 1   # as if v_1 .. v_{l-1} had been folded
        assert native.lib.attnres_layer_sources(ctypes.byref(st), l, out, ctypes.byref(n)) == 0
        got = [out[i] for i in range(n.value)]
        want = []
        for e in O.value_list(l, B, L):
            if e[0] == "embed":
                want.append(h0)
            elif e[0] == "block":
                want.append(reps[e[1] - 1])
            else:
                want.append(partial)
        assert got == want, (l, got, want)


def test_stack_calls_enforce_order(native):
    L, B = 7, 3
    st, *_ = _fake_state(native, L, B)
    out = (ctypes.c_void_p * 128)()
    n = ctypes.c_int()
    # sources of layer 3 need v_1, v_2 folded
    assert native.lib.attnres_layer_sources(ctypes.byref(st), 3, out, ctypes.byref(n)) == native.ATTNRES_ESTATE
    # block_step(2) before block_step(1)
    assert native.lib.attnres_block_step(ctypes.byref(st), 0x999, 2, None, None) == native.ATTNRES_ESTATE
    # F_out may not share memory with the state's rows (h0 at 0x10000, partial at 0x20000)
    assert native.lib.attnres_block_step(ctypes.byref(st), 0x20000 + 8, 1, None, None) == native.ATTNRES_EINVAL
    assert b"F_out overlaps" in native.lib.attnres_last_error()
    assert native.lib.attnres_block_step(ctypes.byref(st), 0x100000, 1, None, None) == native.ATTNRES_EINVAL
    # layer_step: F_prev must be NULL at layer 1; without F_prev layer 2 needs
    # v_1 folded already; with it, layer 3 needs folded == 1
    assert native.lib.attnres_layer_step(ctypes.byref(st), 0x999, 0x888, 1, 0x777, None, None, None) == native.ATTNRES_EINVAL
    assert native.lib.attnres_layer_step(ctypes.byref(st), None, 0x888, 2, 0x777, None, None, None) == native.ATTNRES_ESTATE
    assert native.lib.attnres_layer_step(ctypes.byref(st), 0x999, 0x888, 3, 0x777, None, None, None) == native.ATTNRES_ESTATE
    assert native.lib.attnres_layer_step(ctypes.byref(st), 0x999, 0x888, L + 2, 0x777, None, None, None) == native.ATTNRES_EINVAL
    # out_r may not share memory with the state (rows of 4 x 8 bf16 = 64 B)
    st.folded = 0
    assert native.lib.attnres_layer_step(ctypes.byref(st), None, 0x888, 1, 0x20000, None, None, None) == native.ATTNRES_EINVAL
    assert b"overlaps" in native.lib.attnres_last_error()
    assert native.lib.attnres_layer_step(ctypes.byref(st), None, 0x888, 1, 0x20000 + 48, None, None, None) == native.ATTNRES_EINVAL
    assert native.lib.attnres_layer_step(ctypes.byref(st), None, 0x888, 1, 0x10000 - 32, None, None, None) == native.ATTNRES_EINVAL
    assert st.folded == 0
    assert native.lib.attnres_state_reset(ctypes.byref(st)) == 0


def test_state_resume_sets_progress_only(native):
    # a pipeline stage that starts at layer f + 1 resumes the state at f:
    # the next layer's sources are then those of Eq. 10 after f layers
    L, B = 93, 12
    st, h0, partial, reps = _fake_state(native, L, B)
    out = (ctypes.c_void_p * 128)()
    n = ctypes.c_int()
    for bad in (-1, L + 1):
        assert native.lib.attnres_state_resume(ctypes.byref(st), bad) == native.ATTNRES_EINVAL
        assert st.folded == 0
    for f in (0, 11, 12, 47, 92, 93):
        assert native.lib.attnres_state_resume(ctypes.byref(st), f) == 0 and st.folded == f
        assert native.lib.attnres_layer_sources(ctypes.byref(st), f + 1, out, ctypes.byref(n)) == 0
        assert n.value == O.num_sources(f + 1, B, L)
        # a fused step that folds v_f again is out of order
        if 1 <= f < L:
            assert native.lib.attnres_layer_step(ctypes.byref(st), 0x999, 0x888, f + 1, 0x777, None, None,
                                                 None) == native.ATTNRES_ESTATE
    assert native.lib.attnres_state_resume(None, 3) == native.ATTNRES_EINVAL


def test_interblock_workspace_size_checks_its_arguments(native):
    # host checks before any device query: cached sources 1..9, queries
    # 1..16, a known dtype
    lib = native.lib
    assert lib.attnres_interblock_workspace_size(0, 64, 7168, 1, 12) == native.ATTNRES_ERANGE
    assert lib.attnres_interblock_workspace_size(10, 64, 7168, 1, 12) == native.ATTNRES_ERANGE
    assert lib.attnres_interblock_workspace_size(4, 64, 7168, 1, 17) == native.ATTNRES_ERANGE
    assert lib.attnres_interblock_workspace_size(4, 64, 7168, 7, 12) == native.ATTNRES_EDTYPE
    assert lib.attnres_interblock_workspace_size(4, -1, 7168, 1, 12) == native.ATTNRES_EINVAL


def test_state_init_rejects_bad_arguments(native):
    st = native.AttnresState()
    reps = (ctypes.c_void_p * 3)(0x1000, 0x2000, 0x3000)
    init = native.lib.attnres_state_init
    # rows of 4 x 8 bf16 = 64 bytes: h0 at 0x4000, partial at 0x5000
    assert init(ctypes.byref(st), None, reps, 3, 0x5000, 4, 8, 1, 7, 3, 1e-5) == native.ATTNRES_EINVAL
    assert init(ctypes.byref(st), 0x4000, reps, 2, 0x5000, 4, 8, 1, 7, 3, 1e-5) == native.ATTNRES_EINVAL  # need 3
    assert init(ctypes.byref(st), 0x4000, reps, 3, 0x5000, 4, 8, 7, 7, 3, 1e-5) == native.ATTNRES_EDTYPE
    assert init(ctypes.byref(st), 0x4000, reps, 3, 0x5000, 4, 0, 1, 7, 3, 1e-5) == native.ATTNRES_EINVAL
    assert init(ctypes.byref(st), 0x4000, reps, 3, 0x5000, 4, 8, 1, 7, 3, -1.0) == native.ATTNRES_EINVAL
    # buffers sharing memory: the same address, or overlapping ranges
    assert init(ctypes.byref(st), 0x4000, reps, 3, 0x1000, 4, 8, 1, 7, 3, 1e-5) == native.ATTNRES_EINVAL
    assert init(ctypes.byref(st), 0x4000, reps, 3, 0x4000 + 32, 4, 8, 1, 7, 3, 1e-5) == native.ATTNRES_EINVAL
    assert b"partial overlaps h0" in native.lib.attnres_last_error()
    near = (ctypes.c_void_p * 3)(0x1000, 0x1000 + 48, 0x3000)
    assert init(ctypes.byref(st), 0x4000, near, 3, 0x5000, 4, 8, 1, 7, 3, 1e-5) == native.ATTNRES_EINVAL
    assert b"block_reps[0] overlaps block_reps[1]" in native.lib.attnres_last_error()
    assert st.T == 0 and not st.h0  # a refused call writes nothing
    many = (ctypes.c_void_p * 200)(*range(0x1000, 0x1000 + 200 * 16, 16))
    assert init(ctypes.byref(st), 0x4000, many, 200, 0x5000, 4, 8, 1, 200, 1, 1e-5) == native.ATTNRES_ERANGE
    # adjacent but disjoint buffers are fine
    adj = (ctypes.c_void_p * 3)(0x1000, 0x1040, 0x1080)
    assert init(ctypes.byref(st), 0x4000, adj, 3, 0x4040, 4, 8, 1, 7, 3, 1e-5) == 0


def test_aggregate_rejects_bad_arguments_before_any_launch(native):
    agg = native.lib.attnres_aggregate
    src = (ctypes.c_void_p * 3)(0x1000, 0x2000, 0x3000)
    ok_args = dict(S=3, T=4, d=8, sdt=1, w=0x4000, eps=1e-5, r=0x5000, odt=1)

    def call(**kw):
        a = {**ok_args, **kw}
        return agg(kw.get("src", src), a["S"], a["T"], a["d"], a["sdt"], a["w"], a["eps"], a["r"], a["odt"],
                   None, None, None)

    assert call(S=0) == native.ATTNRES_EINVAL
    assert call(S=129) == native.ATTNRES_ERANGE
    assert call(sdt=5) == native.ATTNRES_EDTYPE
    assert call(odt=-1) == native.ATTNRES_EDTYPE
    assert call(T=-1) == native.ATTNRES_EINVAL
    assert call(d=0) == native.ATTNRES_EINVAL
    assert call(w=None) == native.ATTNRES_EINVAL
    assert call(r=None) == native.ATTNRES_EINVAL
    assert call(eps=float("nan")) == native.ATTNRES_EINVAL
    assert call(eps=-1e-5) == native.ATTNRES_EINVAL
    assert call(T=1 << 40, d=7168) == native.ATTNRES_ERANGE
    assert call(src=(ctypes.c_void_p * 3)(0x1000, None, 0x3000)) == native.ATTNRES_EINVAL
    assert b"sources[1]" in native.lib.attnres_last_error()
    assert agg(None, 3, 4, 8, 1, 0x4000, 1e-5, 0x5000, 1, None, None, None) == native.ATTNRES_EINVAL
    # T = 0 is a valid empty problem: nothing is launched, buffers may be NULL
    assert call(T=0) == 0
    assert agg(None, 3, 0, 8, 1, None, 1e-5, None, 1, None, None, None) == native.ATTNRES_EINVAL  # sources list
    assert agg(src, 3, 0, 8, 1, None, 1e-5, None, 1, None, None, None) == 0


def test_outputs_overlapping_a_source_are_refused(native):
    # [T, d] bf16 sources of 4 x 8 x 2 = 64 bytes at 0x10000 and 0x20000;
    # nothing is dereferenced: the ranges are compared before any launch
    agg = native.lib.attnres_aggregate
    src = (ctypes.c_void_p * 2)(0x10000, 0x20000)

    def call(r, a):
        return agg(src, 2, 4, 8, 1, 0x40000, 1e-5, r, 1, a, None, None)

    assert call(0x10000 + 32, None) == native.ATTNRES_EINVAL        # r inside source 0
    assert b"r overlaps source 0" in native.lib.attnres_last_error()
    assert call(0x20000 - 8, None) == native.ATTNRES_EINVAL         # r's tail reaches source 1
    assert call(0x30000, 0x10000) == native.ATTNRES_EINVAL          # weights on source 0
    assert call(0x30000, 0x30000 + 16) == native.ATTNRES_EINVAL     # weights inside r
    assert b"weights overlap r" in native.lib.attnres_last_error()
    # (every call here is refused before any CUDA call: no launch ever sees
    # these made-up addresses)
    # the host-buffer call checks its host ranges the same way
    host = native.lib.attnres_aggregate_host
    need = native.lib.attnres_aggregate_host_workspace_size(2, 4, 8, 1, 1, 0, 1)
    assert host(src, 2, 4, 8, 1, 0x40000, 1e-5, 0x20000, 1, None, 4, 0x100000, need, None, None) == \
        native.ATTNRES_EINVAL


def test_host_workspace_size_is_the_slot_layout(native):
    # query row, then per slot the [S, chunk, d] sources, r and the weights,
    # each part rounded up to 256 bytes; written out for the K3 block layout
    size = native.lib.attnres_aggregate_host_workspace_size
    q = 7168 * 4                               # 28,672 = 112 x 256
    src = 9 * 256 * 7168 * 2                   # 33,030,144
    r = 256 * 7168 * 2                         # 3,670,016
    a = 256 * 9 * 4                            # 9,216
    assert size(9, 256, 7168, 1, 1, 1, 2) == q + 2 * (src + r + a)
    assert size(9, 256, 7168, 1, 1, 0, 1) == q + src + r
    # fp32 out, ragged sizes: every part padded to 256 bytes on its own
    assert size(3, 5, 10, 0, 0, 1, 3) == 256 + 3 * (768 + 256 + 256)
    assert size(1, 100, 7, 1, 0, 0, 1) == 256 + 1536 + 2816
    assert size(0, 256, 7168, 1, 1, 1, 2) == native.ATTNRES_EINVAL
    assert size(129, 256, 7168, 1, 1, 1, 2) == native.ATTNRES_ERANGE
    assert size(9, 0, 7168, 1, 1, 1, 2) == native.ATTNRES_EINVAL
    assert size(9, 256, 7168, 2, 1, 1, 2) == native.ATTNRES_EDTYPE
    assert size(9, 256, 7168, 1, 1, 2, 2) == native.ATTNRES_EINVAL
    assert size(9, 256, 7168, 1, 1, 1, 0) == native.ATTNRES_EINVAL
    assert size(9, 256, 7168, 1, 1, 1, 9) == native.ATTNRES_EINVAL


def test_aggregate_host_rejects_bad_arguments_before_any_copy(native):
    agg = native.lib.attnres_aggregate_host
    src = (ctypes.c_void_p * 3)(0x1000, 0x2000, 0x3000)
    need = native.lib.attnres_aggregate_host_workspace_size(3, 4, 8, 1, 1, 0, 1)
    ok_args = dict(S=3, T=4, d=8, sdt=1, w=0x4000, eps=1e-5, r=0x5000, odt=1, chunk=4, ws=0x10000, wsb=need)

    def call(**kw):
        a = {**ok_args, **kw}
        return agg(kw.get("src", src), a["S"], a["T"], a["d"], a["sdt"], a["w"], a["eps"], a["r"], a["odt"],
                   None, a["chunk"], a["ws"], a["wsb"], None, None)

    assert call(S=0) == native.ATTNRES_EINVAL
    assert call(S=129) == native.ATTNRES_ERANGE
    assert call(sdt=5) == native.ATTNRES_EDTYPE
    assert call(T=-1) == native.ATTNRES_EINVAL
    assert call(d=0) == native.ATTNRES_EINVAL
    assert call(eps=float("inf")) == native.ATTNRES_EINVAL
    assert call(chunk=0) == native.ATTNRES_EINVAL
    assert call(w=None) == native.ATTNRES_EINVAL
    assert call(r=None) == native.ATTNRES_EINVAL
    assert call(ws=None) == native.ATTNRES_EINVAL
    assert call(ws=0x10010) == native.ATTNRES_EINVAL
    assert b"256-byte" in native.lib.attnres_last_error()
    assert call(wsb=need - 1) == native.ATTNRES_ERANGE
    assert b"one slot" in native.lib.attnres_last_error()
    assert call(src=(ctypes.c_void_p * 3)(0x1000, 0x2000, None)) == native.ATTNRES_EINVAL
    assert b"sources_host[2]" in native.lib.attnres_last_error()
    assert call(T=1 << 40, d=7168) == native.ATTNRES_ERANGE
    # T = 0: nothing copied or launched, buffers may be NULL
    assert agg(src, 3, 0, 8, 1, None, 1e-5, None, 1, None, 4, None, 0, None, None) == 0


def test_backward_rejects_bad_arguments_before_any_launch(native):
    bwd = native.lib.attnres_aggregate_backward
    src = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    grads = (ctypes.c_void_p * 2)(0x3000, 0x4000)
    ok_args = dict(src=src, S=2, T=4, d=8, dt=1, w=0x5000, eps=1e-5, dr=0x6000, g=grads, acc=0, gw=0x7000,
                   ws=0x8000, wsb=1 << 20)

    def call(**kw):
        a = {**ok_args, **kw}
        return bwd(a["src"], a["S"], a["T"], a["d"], a["dt"], a["w"], a["eps"], a["dr"], a["g"], a["acc"], a["gw"],
                   a["ws"], a["wsb"], None, None)

    assert call(S=0) == native.ATTNRES_EINVAL
    assert call(S=129) == native.ATTNRES_ERANGE
    assert call(dt=2) == native.ATTNRES_EDTYPE
    assert call(d=0) == native.ATTNRES_EINVAL
    assert call(gw=None) == native.ATTNRES_EINVAL
    assert call(acc=2) == native.ATTNRES_EINVAL
    assert call(dr=None) == native.ATTNRES_EINVAL
    assert call(ws=None) == native.ATTNRES_EINVAL
    assert call(ws=0x8002) == native.ATTNRES_EINVAL                        # workspace not 4-byte aligned
    assert call(g=(ctypes.c_void_p * 2)(0x3000, 0x1000)) == native.ATTNRES_EINVAL   # grad on a source
    assert b"overlaps sources" in native.lib.attnres_last_error()
    assert call(g=(ctypes.c_void_p * 2)(0x3000, 0x1000 + 40)) == native.ATTNRES_EINVAL   # grad inside a source
    assert call(g=(ctypes.c_void_p * 2)(0x3000, 0x3000)) == native.ATTNRES_EINVAL   # two grads share memory
    assert call(g=(ctypes.c_void_p * 2)(0x3000, 0x3000 + 63)) == native.ATTNRES_EINVAL
    assert call(g=(ctypes.c_void_p * 2)(0x3000, 0x6000 - 8)) == native.ATTNRES_EINVAL   # grad over grad_r
    assert call(src=None) == native.ATTNRES_EINVAL


def test_fold_and_stand_in_backward_reject_bad_arguments(native):
    fold = native.lib.attnres_fold
    assert fold(0x1000, None, 0x2000, 4, 8, 1, None) == native.ATTNRES_EINVAL        # F is NULL
    assert fold(0x1000, 0x3000, None, 4, 8, 1, None) == native.ATTNRES_EINVAL        # dst is NULL
    assert fold(0x1000, 0x3000, 0x2000, 4, 8, 7, None) == native.ATTNRES_EDTYPE
    assert fold(0x1000, 0x3000, 0x2000, -1, 8, 1, None) == native.ATTNRES_EINVAL
    assert fold(None, None, None, 0, 8, 1, None) == 0                                # T = 0: nothing to do
    sb = native.lib.attnres_synthetic_layer_backward
    assert sb(0x1000, 0x2000, 0x3000, None, None, 0x4000, 4, 8, 1, None) == native.ATTNRES_EINVAL
    assert sb(0x1000, None, 0x3000, 0x5000, None, 0x4000, 4, 8, 1, None) == native.ATTNRES_EINVAL
    assert sb(0x1000, 0x2000, 0x3000, 0x5000, None, 0x4000, 4, 8, 3, None) == native.ATTNRES_EDTYPE
    assert sb(0x1000, 0x2000, 0x3000, 0x5000, None, 0x4000, 4, 0, 1, None) == native.ATTNRES_EINVAL


def test_aggregate_fold_rejects_bad_arguments_before_any_launch(native):
    """Fake (never dereferenced) pointers; rows of 4 x 8 bf16 = 64 bytes."""
    af = native.lib.attnres_aggregate_fold
    err = native.lib.attnres_last_error
    srcs = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    prev, F, dst, w, r, a = 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000

    def call(s=srcs, n=2, pv=prev, f=F, ds=dst, T=4, d=8, dt=1, ww=w, eps=1e-5, rr=r, aa=a, flags=0):
        return af(s, n, pv, f, ds, T, d, dt, ww, eps, rr, aa, flags, None, None)

    assert call(f=None) == native.ATTNRES_EINVAL and b"NULL" in err()
    assert call(ds=None) == native.ATTNRES_EINVAL
    assert call(n=-1) == native.ATTNRES_EINVAL
    assert call(n=128) == native.ATTNRES_ERANGE                      # 128 stored + the partial
    assert call(dt=5) == native.ATTNRES_EDTYPE
    assert call(eps=-1.0) == native.ATTNRES_EINVAL
    assert call(flags=2) == native.ATTNRES_EINVAL and b"unknown bits" in err()
    assert call(T=0, s=None, n=0, pv=None, f=None, ds=None, ww=None, rr=None, aa=None) == 0
    # dst may be prev itself (in place) but shares no byte with any other row
    assert call(ds=0x1000 + 32) == native.ATTNRES_EINVAL and b"dst overlaps sources[0]" in err()
    assert call(ds=F) == native.ATTNRES_EINVAL and b"dst overlaps F" in err()
    assert call(ds=prev + 16) == native.ATTNRES_EINVAL and b"dst overlaps prev" in err()
    # outputs share no byte with any row read or written
    for row in (0x2000, prev, F, dst):
        assert call(rr=row + 8) == native.ATTNRES_EINVAL and b"overlaps" in err()
    assert call(aa=F) == native.ATTNRES_EINVAL


def test_debug_wait_test_checks_its_row(native):
    assert native.lib.attnres_debug_wait_test(0, 8) == native.ATTNRES_EINVAL
    assert native.lib.attnres_debug_wait_test(0, -2) == native.ATTNRES_EINVAL
    assert native.lib.attnres_debug_wait_test(0, -1) == 0                           # normal operation
