"""CPU checks of the C ABI: the library loads, exports every function that
include/kda.h declares, and rejects bad arguments on the host before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import linear_attention_layer_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(kda.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return kda.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    declared = _declared_functions()
    assert set(declared) == set(kda.EXPORTED_SYMBOLS), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "KDA_OK"), (1, "KDA_ERR_INVALID_ARGUMENT"), (2, "KDA_ERR_UNSUPPORTED"),
                       (3, "KDA_ERR_CUDA"), (4, "KDA_ERR_TIMEOUT"), (5, "KDA_ERR_DEVICE_CHECK")]:
        assert kda.status_string(code) == name
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"


def test_descriptor_layout_matches_header(tmp_path):
    """The ctypes mirror of kda_desc_t against the C header itself: a small C
    program compiled here prints sizeof and every field's offsetof."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    fields = [f[0] for f in kda.KdaDesc._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"kda.h\"\n"
                   "int main(void) {\n  printf(\"%zu\\n\", sizeof(kda_desc_t));\n" +
                   "".join(f'  printf("%zu\\n", offsetof(kda_desc_t, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", os.path.join(root, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(kda.KdaDesc)
    assert got[1:] == [getattr(kda.KdaDesc, f).offset for f in fields]


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first


def _call_chunk(lib, desc, cu=FAKE, q=FAKE, out=ctypes.c_void_p(0x2000), fn="kda_chunk_fwd"):
    f = getattr(lib, fn)
    return f(ctypes.byref(desc), q, FAKE, FAKE, FAKE, FAKE, None, cu, out, None, None)


@pytest.mark.parametrize("fn", ["kda_chunk_fwd", "kda_recurrent_fwd"])
@pytest.mark.parametrize("bad", [
    dict(dk=48), dict(dv=256), dict(dk=0), dict(num_heads=0), dict(io_dtype=7),
    dict(num_seqs=-1), dict(total_tokens=-5), dict(num_seqs=0, total_tokens=3),
    dict(cu_host=[0, 5, 3]), dict(cu_host=[1, 5, 8]), dict(cu_host=[0, 4, 7]),
])
def test_prefill_rejects_bad_descriptor(lib, fn, bad):
    p = dict(num_seqs=2, total_tokens=8, num_heads=2, dk=64, dv=64, io_dtype=kda.KDA_BF16)
    bad = dict(bad)
    cu_host = bad.pop("cu_host", None)
    p.update(bad)
    desc, keep = kda.make_desc(p["num_seqs"], p["total_tokens"], p["num_heads"], p["dk"], p["dv"],
                               p["io_dtype"], cu_host)
    assert _call_chunk(lib, desc, fn=fn) == 1


def test_prefill_rejects_null_and_aliasing(lib):
    desc, keep = kda.make_desc(2, 8, 2, 64, 64, kda.KDA_BF16, [0, 3, 8])
    assert _call_chunk(lib, desc, cu=None) == 1          # cu_seqlens required
    assert _call_chunk(lib, desc, q=None) == 1           # q required when T > 0
    assert _call_chunk(lib, desc, out=None) == 1         # out required when T > 0
    assert _call_chunk(lib, desc, out=FAKE) == 1         # out aliases q
    assert lib.kda_chunk_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, None,
                             None) == 1


@pytest.mark.parametrize("fn", ["kda_chunk_fwd", "kda_recurrent_fwd", "kda_chunk_fwd_noalloc"])
@pytest.mark.parametrize("every,ckpt,offs", [
    (32, FAKE, FAKE),          # not a multiple of 64
    (-64, FAKE, FAKE),         # negative
    (64, None, FAKE),          # no checkpoint buffer
    (64, FAKE, None),          # no offsets
])
def test_prefill_rejects_bad_checkpoint_arguments(lib, fn, every, ckpt, offs):
    desc, keep = kda.make_desc(2, 8, 2, 64, 64, kda.KDA_BF16, [0, 3, 8])
    desc.checkpoint_every = every
    desc.checkpoints = ckpt
    desc.checkpoint_offsets = offs
    assert _call_chunk(lib, desc, fn=fn) == 1  # KDA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("which", ["initial", "final", "checkpoints"])
def test_recurrent_prefill_rejects_unaligned_states(lib, which):
    """kda_recurrent_fwd moves states and checkpoints four floats at a time:
    one off a 16-byte boundary is refused before anything is enqueued."""
    desc, keep = kda.make_desc(2, 128, 2, 128, 128, kda.KDA_BF16, [0, 64, 128])
    odd = ctypes.c_void_p(0x3004)
    s0 = odd if which == "initial" else None
    fin = odd if which == "final" else None
    if which == "checkpoints":
        desc.checkpoint_every = 64
        desc.checkpoints = odd
        desc.checkpoint_offsets = ctypes.c_void_p(0x5000)
    assert lib.kda_recurrent_fwd(ctypes.byref(desc), FAKE, FAKE, FAKE, FAKE, FAKE, s0, FAKE,
                                 ctypes.c_void_p(0x2000), fin, None) == 1


def test_checkpoint_offsets_count_whole_intervals():
    # lengths 63, 1, 0, 266, 1024
    assert kda.checkpoint_offsets([0, 63, 64, 64, 330, 1354], 64) == [0, 0, 0, 0, 4, 20]


def test_decode_rejects_bad_arguments(lib):
    d, _ = kda.make_desc(4, 4, 2, 128, 128, kda.KDA_BF16)
    f = lib.kda_decode_step
    st = ctypes.c_void_p(0x3000)
    out = ctypes.c_void_p(0x4000)
    assert f(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, None, out, None) == 1  # no state
    assert f(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, st, st, None) == 1     # out == state
    d2, _ = kda.make_desc(4, 5, 2, 128, 128, kda.KDA_BF16)  # total_tokens != num_seqs
    assert f(ctypes.byref(d2), FAKE, FAKE, FAKE, FAKE, FAKE, st, out, None) == 1
    d3, _ = kda.make_desc(4, 4, 2, 96, 128, kda.KDA_BF16)
    assert f(ctypes.byref(d3), FAKE, FAKE, FAKE, FAKE, FAKE, st, out, None) == 1


@pytest.mark.parametrize("window,total,null_q", [(0, 0, False), (2, 7, False), (2, 8, True)])
def test_window_calls_reject_bad_arguments(lib, window, total, null_q):
    d, _ = kda.make_desc(4, total, 2, 128, 128, kda.KDA_BF16)
    q = None if null_q else FAKE
    assert lib.kda_decode_window(ctypes.byref(d), window, q, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 ctypes.c_void_p(0x2000), None) == 1
    assert lib.kda_decode_replay(ctypes.byref(d), window, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 None) == 1


def test_window_rejects_missing_out_and_replay_missing_accept(lib):
    d, _ = kda.make_desc(4, 8, 2, 128, 128, kda.KDA_BF16)
    assert lib.kda_decode_window(ctypes.byref(d), 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None,
                                 None) == 1
    assert lib.kda_decode_window(ctypes.byref(d), 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 None) == 1  # out aliases q
    assert lib.kda_decode_replay(ctypes.byref(d), 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                 None) == 1


def test_fused_window_rejects_unaligned_output_norm_weight(lib):
    """The fused window kernel reads the norm weight four floats at a time, so
    a weight off a 16-byte boundary is refused before anything is enqueued
    (every other argument here passes validation)."""
    d, _ = kda.make_desc(4, 8, 2, 128, 128, kda.KDA_BF16)
    f = kda.KdaFusion(0, None, None, None, None, ctypes.c_void_p(0x1004), 1e-6)
    acc = ctypes.c_void_p(0x1800)
    assert lib.kda_decode_replay_window_fused(
        ctypes.byref(d), ctypes.byref(f), 2, FAKE, FAKE, FAKE, FAKE, FAKE, acc, 2, FAKE, FAKE,
        FAKE, FAKE, FAKE, ctypes.c_void_p(0x3000), ctypes.c_void_p(0x2000), None) == 1


def test_workspace_size_query(lib):
    d, keep = kda.make_desc(1, 65536, 32, 128, 128, kda.KDA_BF16, [0, 65536])
    n = ctypes.c_size_t(123)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value % 256 == 0
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(d), None) == 1
    bad, _ = kda.make_desc(1, 65536, 32, 100, 128, kda.KDA_BF16, [0, 65536])
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1


def _call_bwd(lib, desc, q=FAKE, dq=ctypes.c_void_p(0x2000), d_out=FAKE, cu=FAKE,
              fn="kda_recurrent_bwd"):
    outs = [dq] + [ctypes.c_void_p(0x3000 + 0x1000 * i) for i in range(4)]
    return getattr(lib, fn)(ctypes.byref(desc), q, FAKE, FAKE, FAKE, FAKE, None, cu, d_out,
                            None, *outs, None, None)


@pytest.mark.parametrize("fn", ["kda_recurrent_bwd", "kda_chunk_bwd"])
def test_backward_rejects_bad_arguments(lib, fn):
    _call = lambda *a, **k: _call_bwd(*a, fn=fn, **k)
    cu = [0, 3, 8]
    d, keep = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16, cu)
    assert _call(lib, d) == 1                                   # no workspace
    assert _call(lib, d, cu=None) == 1                          # cu_seqlens required
    assert _call(lib, d, q=None) == 1                           # q required
    assert _call(lib, d, d_out=None) == 1                       # d_out required
    assert _call(lib, d, dq=None) == 1                          # dq required
    assert _call(lib, d, dq=FAKE) == 1                          # dq aliases q
    assert _call(lib, d, q=ctypes.c_void_p(0x1004)) == 1        # not 16-byte aligned
    nohost, keep2 = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16)  # no host cu_seqlens
    assert _call(lib, nohost) == 1
    small, keep3 = kda.make_desc(2, 8, 2, 64, 64, kda.KDA_BF16, cu)
    assert _call(lib, small) == 1                               # supported; no workspace
    d.gate_per_head = 1
    assert _call(lib, d) == 1  # one gate per head is accepted; the workspace is missing
    d.gate_per_head = 3
    assert _call(lib, d) == 1


def test_backward_workspace_size_query(lib):
    d, keep = kda.make_desc(2, 100, 4, 128, 128, kda.KDA_BF16, [0, 60, 100])
    n = ctypes.c_size_t(0)
    assert lib.kda_recurrent_bwd_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    # per resident CTA: one 64 KiB state per 8 tokens of the longest sequence
    # (ceil(60 / 8) = 8) plus a ring of 8
    assert n.value > 0 and n.value % (16 * 64 * 1024) == 0
    nohost, keep2 = kda.make_desc(2, 100, 4, 128, 128, kda.KDA_BF16)
    assert lib.kda_recurrent_bwd_workspace_size(ctypes.byref(nohost), ctypes.byref(n)) == 1


def test_chunk_backward_workspace_size_query(lib):
    d, keep = kda.make_desc(2, 100, 4, 128, 128, kda.KDA_BF16, [0, 60, 100])
    n = ctypes.c_size_t(0)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    # per resident CTA (at most 8 units here): per 16 tokens of the longest
    # sequence (ceil(60 / 16) = 4) one 64 KiB state and a 20 KiB chunk record
    assert n.value > 0 and n.value % (4 * 84 * 1024) == 0
    assert n.value <= 8 * 4 * 84 * 1024
    small, keep3 = kda.make_desc(2, 100, 4, 64, 32, kda.KDA_BF16, [0, 60, 100])
    m = ctypes.c_size_t(0)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(small), ctypes.byref(m)) == 0
    assert m.value > n.value  # the zero-padded copies come on top
    nohost, keep2 = kda.make_desc(2, 100, 4, 128, 128, kda.KDA_BF16)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(nohost), ctypes.byref(n)) == 1


def test_short_conv_rejects_bad_arguments(lib):
    d, keep = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16)
    y = ctypes.c_void_p(0x2000)
    f = lib.kda_short_conv
    assert f(ctypes.byref(d), 0, FAKE, FAKE, None, FAKE, y, None, None) == 1       # width 0
    assert f(ctypes.byref(d), 5, FAKE, FAKE, None, FAKE, y, None, None) == 2       # width 5
    assert f(ctypes.byref(d), 4, FAKE, None, None, FAKE, y, None, None) == 1       # no weight
    assert f(ctypes.byref(d), 4, FAKE, FAKE, None, None, y, None, None) == 1       # no cu_seqlens
    assert f(ctypes.byref(d), 4, None, FAKE, None, FAKE, y, None, None) == 1       # no x
    assert f(ctypes.byref(d), 4, FAKE, ctypes.c_void_p(0x3000), None, FAKE, FAKE, None,
             None) == 1                                                           # y aliases x
    assert f(ctypes.byref(d), 4, ctypes.c_void_p(0x1008), ctypes.c_void_p(0x3000), None, FAKE,
             y, None, None) == 1                                                  # x misaligned
    bad, keep2 = kda.make_desc(2, 8, 2, 48, 48, kda.KDA_BF16)
    assert f(ctypes.byref(bad), 4, FAKE, FAKE, None, FAKE, y, None, None) == 1    # dk = 48


def test_host_prefill_rejects_bad_arguments(lib):
    cu = (ctypes.c_int32 * 3)(0, 3, 8)
    d, keep = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16)
    f = lib.kda_chunk_fwd_host
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, None, cu, ctypes.c_void_p(0x2000), None, None]
    assert f(ctypes.byref(d), 4, *args) == 1                        # no staging area
    d.workspace, d.workspace_bytes = ctypes.c_void_p(0x10000), 1 << 40
    assert f(ctypes.byref(d), 0, *args) == 1                        # groups < 1
    d.checkpoint_every = 64
    assert f(ctypes.byref(d), 4, *args) == 2                        # no checkpoints here
    d.checkpoint_every = 0
    bad = (ctypes.c_int32 * 3)(0, 5, 3)
    assert f(ctypes.byref(d), 4, *args[:6], bad, *args[7:]) == 1    # host cu not monotone
    d.workspace = ctypes.c_void_p(0x10010)                          # not 256-byte aligned
    assert f(ctypes.byref(d), 4, *args) == 1
    n = ctypes.c_size_t(0)
    assert lib.kda_chunk_fwd_host_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    # q, k, v, out bf16 + z fp32 + beta, 8 tokens x 2 heads x 128, two states each way, cu
    assert n.value >= 8 * 2 * 128 * (2 * 4 + 4) + 8 * 2 * 4 + 2 * 2 * 2 * 128 * 128 * 4


def _call_summary(lib, desc, q=FAKE, cu=FAKE, m=ctypes.c_void_p(0x5000),
                  s=ctypes.c_void_p(0x6000)):
    return lib.kda_chunk_fwd_summary(ctypes.byref(desc), q, FAKE, FAKE, FAKE, FAKE, cu, m, s,
                                     None)


def test_summary_rejects_bad_arguments(lib):
    cu = [0, 3, 8]
    d, keep = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16, cu)
    assert _call_summary(lib, d, cu=None) == 1                        # device cu_seqlens
    assert _call_summary(lib, d, q=None) == 1                         # q required
    assert _call_summary(lib, d, m=None) == 1                         # outputs required
    assert _call_summary(lib, d, s=ctypes.c_void_p(0x5000)) == 1      # outputs alias
    assert _call_summary(lib, d, m=FAKE) == 1                         # output aliases q
    assert _call_summary(lib, d, q=ctypes.c_void_p(0x1004)) == 1      # not 16-byte aligned
    nohost, keep2 = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16)    # host copy required
    assert _call_summary(lib, nohost) == 1
    for dk, dv, io in ((64, 64, kda.KDA_BF16), (128, 128, kda.KDA_F32)):
        other, keep3 = kda.make_desc(2, 8, 2, dk, dv, io, cu)
        assert _call_summary(lib, other) == 2                         # KDA_ERR_UNSUPPORTED
    bad_cu, keep4 = kda.make_desc(2, 8, 2, 128, 128, kda.KDA_BF16, [0, 9, 8])
    assert _call_summary(lib, bad_cu) == 1
    n = ctypes.c_size_t(7)
    assert lib.kda_chunk_fwd_summary_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value % 256 == 0
    assert lib.kda_chunk_fwd_summary_workspace_size(ctypes.byref(d), None) == 1


def test_state_scan_rejects_bad_arguments(lib):
    d, keep = kda.make_desc(3, 0, 2, 64, 32, kda.KDA_F32)
    out = ctypes.c_void_p(0x7000)
    scan = lambda dd, count, m=FAKE, s=ctypes.c_void_p(0x2000), o=out: lib.kda_state_scan(
        ctypes.byref(dd), count, m, s, None, o, None)
    assert scan(d, -1) == 1                    # negative count
    assert scan(d, 2, o=None) == 1             # no output
    assert scan(d, 2, m=None) == 1             # transitions needed when count > 0
    assert scan(d, 2, o=FAKE) == 1             # output aliases the transitions
    bad, keep2 = kda.make_desc(3, 0, 2, 48, 32, kda.KDA_F32)
    assert scan(bad, 1) == 1                   # unsupported dk
    empty, keep3 = kda.make_desc(0, 0, 2, 64, 32, kda.KDA_F32)
    assert scan(empty, 2) == 0                 # nothing to do
