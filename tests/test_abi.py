"""The C ABI library builds, loads, exports every declared entry point and
rejects bad arguments on the host (no GPU needed: these paths return before
any CUDA call)."""
import ctypes
import os
import re

import pytest

from hstu_jagged_attention_02_gb300 import binding as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(hstu_[a-z0-9_]+)\s*\(",
                                    src, flags=re.M))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = C.load()
    declared = _declared_functions()
    assert "hstu_attn_fwd" in declared and "hstu_attn_bwd" in declared
    for name in declared:
        assert hasattr(lib, name), name
    assert set(C.EXPORTED) <= set(declared)


def test_struct_sizes_match_the_header():
    # the library checks struct_size; a desc whose struct_size is the ctypes size is accepted
    d = C.make_desc(dtype="bf16", B=2, H=4, d_qk=128, d_v=128, total_tokens=100, max_seq_len=64,
                    alpha=0.1)
    f, b = C.hstu_attn_workspace_size(d)
    assert 0 < f < b
    d.struct_size += 4
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_workspace_size(d)
    assert e.value.status == C.HSTU_ERR_INVALID_ARG


def _desc(**kw):
    base = dict(dtype="bf16", B=3, H=2, d_qk=64, d_v=64, total_tokens=50, max_seq_len=30, alpha=0.125)
    base.update(kw)
    return C.make_desc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), C.HSTU_ERR_INVALID_ARG),
    (dict(H=0), C.HSTU_ERR_INVALID_ARG),
    (dict(total_tokens=-5), C.HSTU_ERR_INVALID_ARG),
    (dict(max_seq_len=0), C.HSTU_ERR_INVALID_ARG),
    (dict(d_qk=96, d_v=96), C.HSTU_ERR_UNSUPPORTED),
    (dict(d_qk=64, d_v=128), C.HSTU_ERR_UNSUPPORTED),
    (dict(dtype="fp32", out_dtype="bf16"), C.HSTU_ERR_UNSUPPORTED),
    (dict(out_dtype="bf16", flags=C.HSTU_FLAG_U_FP32), C.HSTU_ERR_UNSUPPORTED),
    (dict(flags=1 << 7), C.HSTU_ERR_INVALID_ARG),
    (dict(alpha=float("nan")), C.HSTU_ERR_INVALID_ARG),
    (dict(ln_eps=0.0), C.HSTU_ERR_INVALID_ARG),
    (dict(flags=1 << 20), C.HSTU_ERR_INVALID_ARG),
    (dict(num_pos_buckets=0), C.HSTU_ERR_INVALID_ARG),
    (dict(max_seq_len=10**7), C.HSTU_ERR_UNSUPPORTED),
    (dict(dropout_p=1.0), C.HSTU_ERR_INVALID_ARG),
    (dict(dropout_p=-0.25), C.HSTU_ERR_INVALID_ARG),
    (dict(dropout_p=float("nan")), C.HSTU_ERR_INVALID_ARG),
])
def test_descriptor_validation(kw, status):
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_workspace_size(_desc(**kw))
    assert e.value.status == status


def test_workspace_grows_with_tokens():
    f1, b1 = C.hstu_attn_workspace_size(_desc(total_tokens=1000))
    f2, b2 = C.hstu_attn_workspace_size(_desc(total_tokens=2000))
    assert f2 > f1 and b2 > b1
    # backward holds the FP32 dq accumulator and the dO buffer
    assert b2 - f2 >= 2000 * 2 * 64 * (4 + 2)


def test_forward_rejects_bad_arguments_before_any_launch():
    lib = C.load()
    d = _desc()
    args = C.hstu_attn_fwd_args()
    # missing q/k/v/o
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), None, 0, None) == C.HSTU_ERR_INVALID_ARG
    for name in ("seq_offsets", "q", "k", "v", "o"):
        setattr(args, name, 4096)
    # workspace NULL / misaligned / too small
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), None, 0, None) == C.HSTU_ERR_WORKSPACE
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), 4096 + 16, 1 << 20, None) == C.HSTU_ERR_WORKSPACE
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), 4096, 16, None) == C.HSTU_ERR_WORKSPACE
    # misaligned tensor
    args.q = 4096 + 2
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), 4096, 1 << 30, None) == C.HSTU_ERR_INVALID_ARG


def test_backward_requires_du_with_u():
    lib = C.load()
    d = _desc()
    args = C.hstu_attn_bwd_args()
    for name in ("seq_offsets", "q", "k", "v", "o", "dy", "dq", "dk", "dv", "u"):
        setattr(args, name, 4096)
    assert lib.hstu_attn_bwd(ctypes.byref(d), ctypes.byref(args), 4096, 1 << 30, None) == C.HSTU_ERR_INVALID_ARG


def test_plan_keeping_flags_are_checked_before_any_launch():
    lib = C.load()
    d = _desc(total_tokens=1000)
    f, b = C.hstu_attn_workspace_size(d)
    assert b > f
    args = C.hstu_attn_fwd_args()
    for name in ("seq_offsets", "q", "k", "v", "o"):
        setattr(args, name, 4096)
    # keeping the backward's plan takes the backward's workspace
    d.flags = C.HSTU_FLAG_PLAN_BWD
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), 4096, f, None) == C.HSTU_ERR_WORKSPACE
    # each flag belongs to one direction
    d.flags = C.HSTU_FLAG_REUSE_PLAN
    assert lib.hstu_attn_fwd(ctypes.byref(d), ctypes.byref(args), 4096, 1 << 30, None) == C.HSTU_ERR_INVALID_ARG
    bargs = C.hstu_attn_bwd_args()
    for name in ("seq_offsets", "q", "k", "v", "o", "dy", "dq", "dk", "dv"):
        setattr(bargs, name, 4096)
    d.flags = C.HSTU_FLAG_PLAN_BWD
    assert lib.hstu_attn_bwd(ctypes.byref(d), ctypes.byref(bargs), 4096, 1 << 30, None) == C.HSTU_ERR_INVALID_ARG
    # the layer, delta and no-alloc calls plan for themselves
    for flag in (C.HSTU_FLAG_PLAN_BWD, C.HSTU_FLAG_REUSE_PLAN):
        dl = _desc(out_dtype="fp32", total_tokens=1000, flags=flag)
        for call, a in ((C.hstu_layer_fwd, C.hstu_layer_fwd_args()), (C.hstu_layer_bwd, C.hstu_layer_bwd_args()),
                        (C.hstu_attn_fwd_delta, C.hstu_attn_delta_args())):
            if isinstance(a, C.hstu_attn_delta_args):
                a.cand_offsets = a.cache_offsets = 256
                for name in ("q", "k", "v", "o"):
                    setattr(a, name, 4096)
            with pytest.raises(C.HSTUError) as e:
                call(dl, a, 256, 1 << 30, None)
            assert e.value.status == C.HSTU_ERR_INVALID_ARG, (call, flag)
        with pytest.raises(C.HSTUError) as e:
            C.hstu_attn_fwd_noalloc(_desc(total_tokens=1000, flags=flag), args, None)
        assert e.value.status == C.HSTU_ERR_INVALID_ARG


def test_status_strings():
    for s in range(7):
        assert C.hstu_status_string(s) and C.hstu_status_string(s) != "unknown status"
    assert C.hstu_status_string(99) == "unknown status"


def test_layer_descriptor_checks():
    # the layer needs BF16 inputs with FP32 outputs; its workspace holds the
    # attention backward's plus cuBLAS scratch and the layer's own buffers
    ok = _desc(out_dtype="fp32", total_tokens=1000)
    f, b = C.hstu_layer_workspace_size(ok)
    af, ab = C.hstu_attn_workspace_size(ok)
    assert f > af and b > ab and b > f
    for kw in (dict(out_dtype="bf16"), dict(dtype="fp32", out_dtype="fp32")):
        with pytest.raises(C.HSTUError) as e:
            C.hstu_layer_workspace_size(_desc(**kw))
        assert e.value.status == C.HSTU_ERR_UNSUPPORTED


def test_layer_rejects_missing_pointers_before_any_launch():
    d = _desc(out_dtype="fp32", total_tokens=1000)
    args = C.hstu_layer_fwd_args()          # every pointer NULL
    with pytest.raises(C.HSTUError) as e:
        C.hstu_layer_fwd(d, args, 256, 1 << 30, None)
    assert e.value.status == C.HSTU_ERR_INVALID_ARG
    bargs = C.hstu_layer_bwd_args()
    with pytest.raises(C.HSTUError) as e:
        C.hstu_layer_bwd(d, bargs, 256, 1 << 30, None)
    assert e.value.status == C.HSTU_ERR_INVALID_ARG


def test_delta_rejects_missing_pointers_before_any_launch():
    d = _desc(out_dtype="fp32", total_tokens=256)
    args = C.hstu_attn_delta_args()          # every pointer NULL
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_fwd_delta(d, args, 256, 1 << 30, None)
    assert e.value.status == C.HSTU_ERR_INVALID_ARG
    args.cand_offsets = args.cache_offsets = 256   # offsets present, token tensors missing
    args.cache_tokens = -1
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_fwd_delta(d, args, 256, 1 << 30, None)
    assert e.value.status == C.HSTU_ERR_INVALID_ARG


def test_dropout_descriptor_fields():
    f0, b0 = C.hstu_attn_workspace_size(_desc())
    assert C.hstu_attn_workspace_size(_desc(dropout_p=0.5)) == (f0, b0)   # no stored mask
    d = _desc(dropout_p=0.1)
    d.reserved = 1
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_workspace_size(d)
    assert e.value.status == C.HSTU_ERR_INVALID_ARG
    # the seed and offset sit after the pointers of every argument struct
    for cls in (C.hstu_attn_fwd_args, C.hstu_attn_bwd_args, C.hstu_layer_fwd_args, C.hstu_layer_bwd_args):
        names = [n for n, _ in cls._fields_]
        assert names[-2:] == ["dropout_seed", "dropout_offset"], cls
        assert cls.dropout_seed.offset == 8 * (len(names) - 2)


def test_delta_rejects_dropout():
    d = _desc(out_dtype="fp32", total_tokens=256, dropout_p=0.1)
    args = C.hstu_attn_delta_args()
    args.cand_offsets = args.cache_offsets = 256
    with pytest.raises(C.HSTUError) as e:
        C.hstu_attn_fwd_delta(d, args, 256, 1 << 30, None)
    assert e.value.status == C.HSTU_ERR_UNSUPPORTED
