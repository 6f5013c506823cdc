"""CPU-only checks of the C ABI: the library builds, loads and exports every symbol that
include/pa.h declares, and host-checkable argument errors are rejected before any CUDA call
(no compute runs here)."""
import ctypes
import os
import re
import shutil

import pytest

from paged_kv_cache_238_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    os.path.join(ROOT, "paged_kv_cache_238_gb300", "libpa.so")), reason="needs nvcc to build libpa")

FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced by these calls


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = B.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings():
    assert B.status_string(B.PA_OK) == "PA_OK"
    assert B.status_string(B.PA_ERR_INVALID_ARG) == "PA_ERR_INVALID_ARG"
    assert B.status_string(B.PA_ERR_UNSUPPORTED) == "PA_ERR_UNSUPPORTED"
    assert B.status_string(B.PA_ERR_CUDA) == "PA_ERR_CUDA"
    assert B.status_string(99) == "PA_UNKNOWN_STATUS"


def _decode(lib, **kw):
    args = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, lens=FAKE, S=2, max_len=64, Hq=8, Hkv=2,
                D=128, NB=16, scale=0.1, dt=B.PA_BF16, ws=FAKE, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.pa_decode(args["out"], args["q"], args["kc"], args["vc"], args["bt"], args["mb"], args["lens"],
                         args["S"], args["max_len"], args["Hq"], args["Hkv"], args["D"], args["NB"], args["scale"],
                         args["dt"], args["ws"], args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(Hq=6, Hkv=4), B.PA_ERR_INVALID_ARG),           # q heads not a multiple of kv heads
    (dict(Hkv=0), B.PA_ERR_INVALID_ARG),
    (dict(D=96), B.PA_ERR_UNSUPPORTED),                    # head_dim outside {64, 128}
    (dict(D=0), B.PA_ERR_INVALID_ARG),
    (dict(dt=7), B.PA_ERR_INVALID_ARG),
    (dict(q=None), B.PA_ERR_INVALID_ARG),
    (dict(bt=None), B.PA_ERR_INVALID_ARG),
    (dict(out=FAKE + 8), B.PA_ERR_INVALID_ARG),            # misaligned
    (dict(lens=FAKE + 2), B.PA_ERR_INVALID_ARG),           # misaligned int32 array
    (dict(max_len=65), B.PA_ERR_INVALID_ARG),              # beyond max_blocks * 16
    (dict(S=-1), B.PA_ERR_INVALID_ARG),
    (dict(NB=0), B.PA_ERR_INVALID_ARG),
    (dict(NB=1 << 27, Hkv=2), B.PA_ERR_UNSUPPORTED),       # pool rows beyond 32-bit coordinates
])
def test_decode_rejects_bad_arguments(kw, expect):
    assert _decode(B.load(), **kw) == expect


def test_decode_zero_sequences_is_a_no_op():
    assert _decode(B.load(), S=0, out=None, q=None) == B.PA_OK


@pytest.mark.parametrize("kw,expect", [
    (dict(T=-1), B.PA_ERR_INVALID_ARG),
    (dict(H=0), B.PA_ERR_INVALID_ARG),
    (dict(D=12), B.PA_ERR_UNSUPPORTED),                    # row not a multiple of 16 bytes (bf16)
    (dict(slots=None), B.PA_ERR_INVALID_ARG),
    (dict(slots=FAKE + 4), B.PA_ERR_INVALID_ARG),
    (dict(k=FAKE + 2), B.PA_ERR_INVALID_ARG),
    (dict(dt=5), B.PA_ERR_INVALID_ARG),
    (dict(T=0, k=None), B.PA_OK),                          # nothing to write
])
def test_reshape_rejects_bad_arguments(kw, expect):
    a = dict(k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, slots=FAKE, T=4, H=2, D=128, NB=8, dt=B.PA_BF16)
    a.update(kw)
    assert B.load().pa_reshape_and_cache(a["k"], a["v"], a["kc"], a["vc"], a["slots"], a["T"], a["H"], a["D"],
                                         a["NB"], a["dt"], None) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(max_chunk=65), B.PA_ERR_INVALID_ARG),            # chunk longer than any sequence may be
    (dict(qsl=None), B.PA_ERR_INVALID_ARG),
    (dict(max_chunk=-1), B.PA_ERR_INVALID_ARG),
    (dict(D=80), B.PA_ERR_UNSUPPORTED),
    (dict(max_chunk=0, q=None), B.PA_OK),
])
def test_prefill_rejects_bad_arguments(kw, expect):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, lens=FAKE, qsl=FAKE, S=2, max_chunk=16,
             max_len=64, Hq=8, Hkv=2, D=128, NB=16, dt=B.PA_BF16)
    a.update(kw)
    assert B.load().pa_prefill_chunk(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["lens"], a["qsl"],
                                     a["S"], a["max_chunk"], a["max_len"], a["Hq"], a["Hkv"], a["D"], a["NB"],
                                     0.1, a["dt"], None) == expect


def test_workspace_size_of_invalid_shape_is_zero():
    assert B.load().pa_decode_workspace_size(2, 6, 4, 128, 64, B.PA_BF16) == 0


def test_device_errors_needs_an_output_pointer():
    assert B.load().pa_get_device_errors(None, 0) == B.PA_ERR_INVALID_ARG


def test_product_path_does_not_reference_the_oracle():
    """The CUDA library and its binding never load, link or import the oracle."""
    pkg = os.path.join(ROOT, "paged_kv_cache_238_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "pa_oracle" not in text, f
    with open(os.path.join(ROOT, "include", "pa.h")) as fh:
        assert "oracle" not in fh.read()


def test_library_does_not_link_the_oracle():
    lib = B.load()
    for sym in ("oracle_attention", "oracle_reshape_and_cache"):
        with pytest.raises(AttributeError):
            getattr(lib, sym)
    assert isinstance(lib, ctypes.CDLL)


def _decode_bs(lib, bs, **kw):
    args = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, lens=FAKE, S=2, max_len=64, Hq=8, Hkv=2,
                D=128, NB=16, scale=0.1, dt=B.PA_BF16, ws=FAKE, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.pa_decode_bs(args["out"], args["q"], args["kc"], args["vc"], args["bt"], args["mb"], args["lens"],
                            args["S"], args["max_len"], args["Hq"], args["Hkv"], args["D"], args["NB"], bs,
                            args["scale"], args["dt"], args["ws"], args["ws_bytes"], args["stream"])


@pytest.mark.parametrize("bs,kw,expect", [
    (48, {}, B.PA_ERR_UNSUPPORTED),                      # not a power of two in 16..128
    (256, {}, B.PA_ERR_UNSUPPORTED),
    (8, {}, B.PA_ERR_UNSUPPORTED),
    (0, {}, B.PA_ERR_INVALID_ARG),
    (-16, {}, B.PA_ERR_INVALID_ARG),
    (32, dict(max_len=129), B.PA_ERR_INVALID_ARG),        # beyond max_blocks * 32
    (128, dict(NB=1 << 23, Hkv=2), B.PA_ERR_UNSUPPORTED),  # pool rows beyond 32-bit coordinates
    (64, dict(S=0, out=None, q=None), B.PA_OK),
])
def test_decode_bs_checks_the_block_size(bs, kw, expect):
    assert _decode_bs(B.load(), bs, **kw) == expect


@pytest.mark.parametrize("bs,expect", [(48, B.PA_ERR_UNSUPPORTED), (0, B.PA_ERR_INVALID_ARG)])
def test_other_bs_entry_points_check_the_block_size(bs, expect):
    lib = B.load()
    assert lib.pa_reshape_and_cache_bs(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 8, bs, B.PA_BF16, None) == expect
    assert lib.pa_copy_blocks_bs(FAKE, FAKE, FAKE, 2, 2, 128, 8, bs, B.PA_BF16, None) == expect
    assert lib.pa_prefill_chunk_bs(FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 16, 64, 8, 2, 128, 16, bs, 0.1,
                                   B.PA_BF16, None) == expect


def test_step_desc_layout_matches_the_header(tmp_path):
    """The binding's ctypes mirror of pa_step_desc has the C layout (offsets from gcc)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("needs gcc")
    names = [f[0] for f in B.StepDesc._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "pa.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(pa_step_desc));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(pa_step_desc, {n}));\n' for n in names) + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(B.StepDesc)] + [getattr(B.StepDesc, n).offset for n in names]
    assert got == want


def _step(**kw):
    d = B.StepDesc()
    base = dict(k_cache=FAKE, v_cache=FAKE, num_blocks=64, block_size=16, num_q_heads=8, num_kv_heads=2,
                head_dim=128, scale=0.1, dtype=B.PA_BF16,
                decode_out=FAKE, decode_q=FAKE, decode_block_table=FAKE, decode_max_blocks_per_seq=4,
                decode_seq_lens=FAKE, num_decode_seqs=2, decode_max_seq_len=64, workspace=FAKE,
                workspace_bytes=1 << 24,
                prefill_out=FAKE, prefill_q=FAKE, prefill_block_table=FAKE, prefill_max_blocks_per_seq=4,
                prefill_seq_lens=FAKE, query_start_loc=FAKE, num_prefill_seqs=2, max_chunk_len=16,
                prefill_max_seq_len=64, k_new=FAKE, v_new=FAKE, slot_mapping=FAKE, num_new_tokens=4)
    base.update(kw)
    for k, v in base.items():
        setattr(d, k, v)
    return B.load().pa_step(ctypes.byref(d), None)


@pytest.mark.parametrize("kw,expect", [
    (dict(decode_sms=-1), B.PA_ERR_INVALID_ARG),
    (dict(num_decode_seqs=-1), B.PA_ERR_INVALID_ARG),
    (dict(head_dim=96), B.PA_ERR_UNSUPPORTED),
    (dict(block_size=48), B.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), B.PA_ERR_INVALID_ARG),
    (dict(decode_q=None), B.PA_ERR_INVALID_ARG),                 # a part's own checks still apply
    (dict(query_start_loc=None), B.PA_ERR_INVALID_ARG),
    (dict(slot_mapping=FAKE + 4), B.PA_ERR_INVALID_ARG),
    (dict(prefill_max_seq_len=65), B.PA_ERR_INVALID_ARG),        # beyond 4 blocks of 16
    (dict(num_new_tokens=0, num_prefill_seqs=0, num_decode_seqs=0, k_cache=None), B.PA_OK),  # nothing to do
    (dict(num_new_tokens=0, num_prefill_seqs=0, num_decode_seqs=0, prefill_max_blocks_per_seq=0,
          decode_max_blocks_per_seq=0), B.PA_OK),              # skipped parts are not checked
])
def test_step_rejects_bad_arguments(kw, expect):
    assert _step(**kw) == expect


def test_step_null_descriptor():
    assert B.load().pa_step(None, None) == B.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,expect", [
    (dict(k_new=None), B.PA_ERR_INVALID_ARG),
    (dict(slots=FAKE + 4), B.PA_ERR_INVALID_ARG),       # int64 slots must be 8-byte aligned
    (dict(v_new=FAKE + 8), B.PA_ERR_INVALID_ARG),
    (dict(bs=48), B.PA_ERR_UNSUPPORTED),
    (dict(D=96), B.PA_ERR_UNSUPPORTED),
    (dict(max_len=65), B.PA_ERR_INVALID_ARG),
    (dict(S=0, out=None, q=None, k_new=None), B.PA_OK),
    (dict(flags=4), B.PA_ERR_INVALID_ARG),               # unknown flag bit
])
def test_decode_append_rejects_bad_arguments(kw, expect):
    a = dict(out=FAKE, q=FAKE, k_new=FAKE, v_new=FAKE, slots=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, mb=4, lens=FAKE, S=2,
             max_len=64, Hq=8, Hkv=2, D=128, NB=16, bs=16, dt=B.PA_BF16)
    a.update(kw)
    assert B.load().pa_decode_append(a["out"], a["q"], a["k_new"], a["v_new"], a["slots"], a["kc"], a["vc"], a["bt"],
                                     a["mb"], a["lens"], a["S"], a["max_len"], a["Hq"], a["Hkv"], a["D"], a["NB"],
                                     a["bs"], 0.1, a["dt"], FAKE, 1 << 24, a.get("flags", 0), None) == expect


def test_wait_drill_arguments_are_checked_on_the_host():
    """The wait-drill hook only sets host-side state: unknown kinds and limits outside
    1 us .. 1 s are rejected, valid settings are taken and PA_DRILL_OFF restores normal
    operation (no kernel runs here)."""
    lib = B.load()
    assert lib.pa_debug_set_wait_drill(3, 2_000_000) == B.PA_ERR_INVALID_ARG
    assert lib.pa_debug_set_wait_drill(-1, 2_000_000) == B.PA_ERR_INVALID_ARG
    assert lib.pa_debug_set_wait_drill(B.PA_DRILL_DECODE_STAGE, 999) == B.PA_ERR_INVALID_ARG
    assert lib.pa_debug_set_wait_drill(B.PA_DRILL_DECODE_STAGE, 1_000_000_001) == B.PA_ERR_INVALID_ARG
    try:
        assert lib.pa_debug_set_wait_drill(B.PA_DRILL_DECODE_STAGE, 2_000_000) == B.PA_OK
        assert lib.pa_debug_set_wait_drill(B.PA_DRILL_PREFILL_K_TILE, 1000) == B.PA_OK
    finally:
        assert lib.pa_debug_set_wait_drill(B.PA_DRILL_OFF, 0) == B.PA_OK


@pytest.mark.parametrize("kw,expect", [
    (dict(prefix=0), B.PA_ERR_INVALID_ARG),            # no prefix
    (dict(prefix=24), B.PA_ERR_INVALID_ARG),           # not a whole number of 16-token blocks
    (dict(prefix=2048, msl=1024), B.PA_ERR_INVALID_ARG),  # longer than every sequence may be
    (dict(Hq=16, Hkv=8), B.PA_ERR_UNSUPPORTED),         # 2 q heads per kv head
    (dict(D=64), B.PA_ERR_UNSUPPORTED),                 # head_dim 64
    (dict(dt_ok=False), B.PA_ERR_INVALID_ARG),          # unaligned output
    (dict(flags=4), B.PA_ERR_INVALID_ARG),              # unknown flag bit
])
def test_shared_prefix_decode_rejects_bad_arguments(kw, expect):
    """Host checks of pa_decode_shared_prefix, made before anything touches a device."""
    lib = B.load()
    S, Hq, Hkv, D, msl = 4, kw.get("Hq", 32), kw.get("Hkv", 8), kw.get("D", 128), kw.get("msl", 2048)
    out = FAKE if kw.get("dt_ok", True) else FAKE + 2
    st = lib.pa_decode_shared_prefix(out, FAKE, FAKE, FAKE, FAKE, msl // 16, FAKE, S, msl, Hq, Hkv, D, 4096,
                                     ctypes.c_float(0.1), kw.get("prefix", 1024), FAKE, 1 << 30, kw.get("flags", 0), None)
    assert st == expect
