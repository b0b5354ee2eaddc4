"""The C-ABI library loads, exports what include/pkv.h declares, and its host checks hold.

No kernel is launched here: every call below is rejected by a host-side check
that runs before the library touches a device.
"""
import ctypes
import os
import re

import pytest

from paged_kv_cache_256_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(pkv_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["pkv_paged_decode_attn", "pkv_paged_decode_attn_workspace_size", "pkv_kv_append",
              "pkv_check_error", "pkv_kv_bytes", "pkv_status_string", "pkv_version"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_binding_exposes_same_names():
    import paged_kv_cache_256_gb300 as pkg
    for name in declared_functions():
        assert hasattr(pkg, name), name


def test_header_constants_match_the_binding():
    """Every numeric #define PKV_... of the header has the same value in the binding."""
    import paged_kv_cache_256_gb300 as pkg
    text = open(HEADER).read()
    defs = re.findall(r"^#define\s+(PKV_\w+)\s+(0x[0-9A-Fa-f]+|\d+)u?\b", text, flags=re.M)
    assert len(defs) >= 10
    for name, value in defs:
        assert getattr(_lib, name) == int(value, 0), name
        assert getattr(pkg, name, getattr(_lib, name)) == int(value, 0), name


def test_status_strings(lib):
    for code in range(8):
        assert _lib.status_name(code).startswith("PKV_")
    assert _lib.status_name(_lib.PKV_ERR_TIMEOUT) == "PKV_ERR_TIMEOUT"
    assert _lib.status_name(99) == "PKV_ERR_UNKNOWN"


def test_version(lib):
    assert lib.pkv_version() >= 10000


def test_kv_bytes_matches_pages(lib):
    from tests.oracle_pins import _golden_rows
    for name, L, n_kv, d, p, tokens, expected in _golden_rows():
        assert lib.pkv_kv_bytes(L, n_kv, d, p, tokens) == expected, name
    assert lib.pkv_kv_bytes(-1, 8, 128, 2, 1) == -1


FAKE = 0x10000  # a 64 KiB-aligned non-null address that is never dereferenced


def attn(lib, **over):
    args = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, num_seqs=2, q_len=1, n_q=4, n_kv=2,
                head_dim=64, block_size=16, max_blocks=3, num_blocks=8, scale=0.125, out=FAKE,
                out_dtype=0, ws=FAKE, ws_bytes=1 << 20, flags=0, stream=None)
    args.update(over)
    return lib.pkv_paged_decode_attn(
        args["q"], args["k"], args["v"], args["bt"], args["cl"], args["num_seqs"], args["q_len"],
        args["n_q"], args["n_kv"], args["head_dim"], args["block_size"], args["max_blocks"],
        args["num_blocks"], args["scale"], args["out"], args["out_dtype"], args["ws"],
        args["ws_bytes"], args["flags"], args["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(n_q=6, n_kv=4), _lib.PKV_ERR_INVALID_ARG),     # n_q % n_kv != 0
    (dict(n_kv=0), _lib.PKV_ERR_INVALID_ARG),
    (dict(num_seqs=-1), _lib.PKV_ERR_INVALID_ARG),
    (dict(q_len=0), _lib.PKV_ERR_INVALID_ARG),
    (dict(head_dim=96), _lib.PKV_ERR_UNSUPPORTED),
    (dict(head_dim=256), _lib.PKV_ERR_UNSUPPORTED),
    (dict(block_size=8), _lib.PKV_ERR_UNSUPPORTED),
    (dict(block_size=64), _lib.PKV_ERR_UNSUPPORTED),
    (dict(q_len=(1 << 16) + 1), _lib.PKV_ERR_UNSUPPORTED),      # beyond the largest chunk
    (dict(n_q=1024, n_kv=1, q_len=1 << 15), _lib.PKV_ERR_UNSUPPORTED),  # > 2^24 rows per KV head
    (dict(out_dtype=2), _lib.PKV_ERR_INVALID_ARG),
    (dict(max_blocks=0), _lib.PKV_ERR_INVALID_ARG),
    (dict(num_blocks=0), _lib.PKV_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.PKV_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _lib.PKV_ERR_INVALID_ARG),
    (dict(q=None), _lib.PKV_ERR_INVALID_ARG),
    (dict(k=None), _lib.PKV_ERR_INVALID_ARG),
    (dict(bt=None), _lib.PKV_ERR_INVALID_ARG),
    (dict(cl=None), _lib.PKV_ERR_INVALID_ARG),
    (dict(out=None), _lib.PKV_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), _lib.PKV_ERR_INVALID_ARG),        # bf16 tensors need 16-byte alignment
    (dict(out=FAKE + 4), _lib.PKV_ERR_INVALID_ARG),
    (dict(bt=FAKE + 2), _lib.PKV_ERR_INVALID_ARG),
    (dict(num_blocks=1 << 30, n_q=8, n_kv=8), _lib.PKV_ERR_UNSUPPORTED),  # cache view over 2^31 rows
])
def test_attn_host_checks(lib, over, status):
    assert attn(lib, **over) == status


def test_attn_empty_batch_is_a_noop(lib):
    assert attn(lib, num_seqs=0, q=None, out=None, ws=None) == _lib.PKV_OK


def kv_append(lib, **over):
    args = dict(kn=FAKE, vn=FAKE, sm=FAKE, T=4, n_kv=2, d=64, bs=16, nb=8, kc=FAKE, vc=FAKE,
                flags=0, stream=None)
    args.update(over)
    return lib.pkv_kv_append(args["kn"], args["vn"], args["sm"], args["T"], args["n_kv"], args["d"],
                             args["bs"], args["nb"], args["kc"], args["vc"], args["flags"],
                             args["stream"])


@pytest.mark.parametrize("over", [
    dict(T=-1), dict(n_kv=0), dict(d=12), dict(d=4), dict(bs=0), dict(nb=0), dict(kn=None),
    dict(vc=None), dict(sm=None), dict(kn=FAKE + 8), dict(sm=FAKE + 1),
])
def test_append_host_checks(lib, over):
    assert kv_append(lib, **over) == _lib.PKV_ERR_INVALID_ARG


def test_append_zero_tokens_is_a_noop(lib):
    assert kv_append(lib, T=0, kn=None, vn=None, sm=None) == _lib.PKV_OK


def test_workspace_size_rejects_bad_shapes(lib):
    assert lib.pkv_paged_decode_attn_workspace_size(2, 1, 6, 4, 64, 16, 100, 0) == 0
    assert lib.pkv_paged_decode_attn_workspace_size(2, 1, 4, 2, 96, 16, 100, 0) == 0


def test_check_error_rejects_null(lib):
    assert lib.pkv_check_error(None, None) == _lib.PKV_ERR_INVALID_ARG


def test_product_sources_do_not_reach_the_oracle():
    """Neither the CUDA sources nor the binding name the CPU oracle."""
    import glob
    pkg = os.path.dirname(_lib.__file__)
    files = glob.glob(os.path.join(pkg, "csrc", "*")) + glob.glob(os.path.join(pkg, "*.py"))
    for f in files:
        text = open(f).read()
        for pat in (r"^\s*(from|import)\s+oracle\b", r"\boracle_\w+\s*\(", r"pkv_oracle"):
            assert not re.search(pat, text, flags=re.M), (f, pat)


def test_params_struct_layout_matches_header(tmp_path):
    """The ctypes mirror of pkv_attn_params has the C compiler's size and offsets."""
    fields = [f for f, _ in _lib.pkv_attn_params._fields_]
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "pkv.h"\nint main(void) {\n'
        '  printf("%zu\\n", sizeof(pkv_attn_params));\n' +
        "".join(f'  printf("%zu\\n", offsetof(pkv_attn_params, {f}));\n' for f in fields) +
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_lib.pkv_attn_params)
    for f, off in zip(fields, got[1:]):
        assert getattr(_lib.pkv_attn_params, f).offset == off, f


def _params(**over):
    p = _lib.pkv_attn_params(q=FAKE, k_cache=FAKE, v_cache=FAKE, block_tables=FAKE,
                             context_lens=FAKE, num_seqs=0, q_len=1, n_q=4, n_kv=2, head_dim=64,
                             block_size=16, max_blocks_per_seq=3, num_blocks=8, scale=0.125,
                             out=FAKE, out_dtype=0, workspace=FAKE, workspace_bytes=1 << 20,
                             flags=0, window=0)
    for k, v in over.items():
        setattr(p, k, v)
    return p


def test_params_entry_host_checks(lib):
    assert lib.pkv_paged_decode_attn_ex(None, None) == _lib.PKV_ERR_INVALID_ARG
    # num_seqs == 0 is accepted without touching a device ...
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params()), None) == _lib.PKV_OK
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params(window=5)), None) == _lib.PKV_OK
    # ... after every argument check, so a bad window or shape is still refused.
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params(window=-1)),
                                        None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params(n_q=3)),
                                        None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params(head_dim=96)),
                                        None) == _lib.PKV_ERR_UNSUPPORTED
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params(kv_dtype=3)),
                                        None) == _lib.PKV_ERR_INVALID_ARG
    # per-block scales: the scale tensor is required and 16-byte aligned
    blk = _lib.PKV_KV_FP8_E4M3_BLOCK
    assert lib.pkv_paged_decode_attn_ex(
        ctypes.byref(_params(num_seqs=2, kv_dtype=blk, v_cache=None)),
        None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_decode_attn_ex(
        ctypes.byref(_params(num_seqs=2, kv_dtype=blk, v_cache=None, kv_scales=FAKE + 8)),
        None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_decode_attn_ex(ctypes.byref(_params(kv_dtype=blk)), None) == _lib.PKV_OK
    # an 8-bit cache needs its scales and no V pointer (checked before any device call)
    assert lib.pkv_paged_decode_attn_ex(
        ctypes.byref(_params(num_seqs=2, kv_dtype=_lib.PKV_KV_FP8_E4M3)),
        None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_decode_attn_ex(
        ctypes.byref(_params(num_seqs=2, kv_dtype=_lib.PKV_KV_FP8_E4M3, k_scale=FAKE,
                             v_scale=FAKE)), None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_paged_decode_attn_ex(
        ctypes.byref(_params(kv_dtype=_lib.PKV_KV_FP8_E4M3)), None) == _lib.PKV_OK


def test_fp8_block_append_and_copy_host_checks(lib):
    args = [FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, FAKE, None, 0, None]
    assert lib.pkv_kv_append_fp8_block(*args) == _lib.PKV_ERR_INVALID_ARG  # null kv_scales
    args[9] = FAKE + 4
    assert lib.pkv_kv_append_fp8_block(*args) == _lib.PKV_ERR_INVALID_ARG  # misaligned scales
    args[9] = FAKE
    args[5] = 60
    assert lib.pkv_kv_append_fp8_block(*args) == _lib.PKV_ERR_INVALID_ARG  # head_dim % 8
    args[5], args[3] = 64, 0
    assert lib.pkv_kv_append_fp8_block(*args) == _lib.PKV_OK  # nothing to append
    # block scales need the 8-bit flag and a scale tensor in place of v_cache
    both = _lib.PKV_FLAG_KV_FP8 | _lib.PKV_FLAG_KV_BLOCK_SCALES
    assert lib.pkv_copy_blocks(FAKE, FAKE, FAKE, 1, 8, 2, 64, 16, _lib.PKV_FLAG_KV_BLOCK_SCALES,
                               None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(FAKE, None, FAKE, 1, 8, 2, 64, 16, both,
                               None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(FAKE, FAKE, FAKE, 0, 8, 2, 64, 16, both, None) == _lib.PKV_OK


def test_fp8_append_and_copy_host_checks(lib):
    args = [FAKE, FAKE, FAKE, 4, 2, 64, 16, 8, None, FAKE, FAKE, 0, None]
    assert lib.pkv_kv_append_fp8(*args) == _lib.PKV_ERR_INVALID_ARG  # null k_scale
    args[8] = FAKE
    args[5] = 60  # head_dim not a multiple of 8
    assert lib.pkv_kv_append_fp8(*args) == _lib.PKV_ERR_INVALID_ARG
    args[5], args[3] = 64, 0
    assert lib.pkv_kv_append_fp8(*args) == _lib.PKV_OK  # nothing to append
    # an interleaved 8-bit cache has no separate V pointer; bf16 caches need one
    assert lib.pkv_copy_blocks(FAKE, FAKE, FAKE, 1, 8, 2, 64, 16, _lib.PKV_FLAG_KV_FP8,
                               None) == _lib.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy_blocks(FAKE, None, FAKE, 1, 8, 2, 64, 16, 0,
                               None) == _lib.PKV_ERR_INVALID_ARG
