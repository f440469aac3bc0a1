"""C ABI checks that need no GPU: the library loads, exports every function
include/xqa.h declares, the ctypes struct matches the C layout, and host-side
validation rejects malformed arguments before any CUDA call."""

import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_decode_20_gb300 import build as B
from paged_kv_decode_20_gb300 import xqa as X

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xqa.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return X.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(xqa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(X.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", X.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (xqa_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_params_struct_layout_matches_c(tmp_path):
    fields = [f for f, _ in X.XqaParams._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "xqa.h"', "int main(void){",
            'printf("%zu\\n", sizeof(xqa_params));']
    prog += [f'printf("%zu\\n", offsetof(xqa_params, {f}));' for f in fields]
    prog += ["return 0;}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I" + os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(X.XqaParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(X.XqaParams, f).offset == off, f


def test_status_strings(lib):
    assert X.status_name(X.XQA_OK) == "XQA_OK"
    assert X.status_name(X.XQA_ERR_WORKSPACE_TOO_SMALL) == "XQA_ERR_WORKSPACE_TOO_SMALL"
    assert X.status_name(99) == "XQA_ERR_UNKNOWN"


def fake_params(**over):
    """A well-formed parameter block with fake (never dereferenced) pointers."""
    p = X.XqaParams()
    fake = 0x10000
    p.q = p.k_cache = p.v_cache = p.page_table = p.seq_lens = p.output = fake
    p.q_dtype = p.kv_dtype = p.out_dtype = X.XQA_BF16
    p.kv_layout = X.XQA_NHD
    p.num_pages = 128
    p.pages_per_seq = 8
    p.batch_size, p.num_q_heads, p.num_kv_heads = 4, 32, 8
    p.head_dim, p.page_size, p.q_seq_len = 128, 64, 1
    p.q_scale = p.kv_scale = p.rcp_out_scale = 1.0
    for k, v in over.items():
        setattr(p, k, v)
    return p


BAD = [
    (dict(page_size=48), X.XQA_ERR_INVALID_ARG, "page_size"),
    (dict(num_q_heads=30), X.XQA_ERR_INVALID_ARG, "multiple"),
    (dict(batch_size=0), X.XQA_ERR_INVALID_ARG, "batch_size"),
    (dict(q=0), X.XQA_ERR_INVALID_ARG, "required"),
    (dict(q_seq_len=0), X.XQA_ERR_INVALID_ARG, "q_seq_len"),
    (dict(q_seq_len=33), X.XQA_ERR_UNSUPPORTED, "q_seq_len"),
    (dict(sliding_win_size=-1), X.XQA_ERR_INVALID_ARG, "sliding"),
    (dict(q_dtype=X.XQA_E4M3, out_dtype=X.XQA_E4M3), X.XQA_ERR_INVALID_ARG, "q dtype"),
    (dict(kv_dtype=X.XQA_F16), X.XQA_ERR_INVALID_ARG, "kv dtype"),
    (dict(out_dtype=X.XQA_F16), X.XQA_ERR_UNSUPPORTED, "output dtype"),
    (dict(out_dtype=X.XQA_E4M3), X.XQA_ERR_UNSUPPORTED, "fp8 cache"),
    (dict(head_dim=96), X.XQA_ERR_UNSUPPORTED, "head_dim"),
    (dict(kv_dtype=X.XQA_E4M3, head_dim=64), X.XQA_ERR_UNSUPPORTED, "head_dim"),
    (dict(k_cache=0x10008), X.XQA_ERR_INVALID_ARG, "16-byte"),
    (dict(pages_per_seq=0), X.XQA_ERR_INVALID_ARG, "pages_per_seq"),
    (dict(num_pages=1 << 28), X.XQA_ERR_UNSUPPORTED, "32-bit"),
]


@pytest.mark.parametrize("over,status,text", BAD, ids=[t for _, _, t in BAD])
def test_validation_rejects_before_launch(lib, over, status, text):
    p = fake_params(**over)
    st = lib.xqa_decode(ctypes.byref(p), None, 0, None, None)
    assert st == status
    assert text in lib.xqa_last_error().decode()
    assert lib.xqa_workspace_size(ctypes.byref(p), 152) == ctypes.c_size_t(-1).value


def test_null_params_rejected(lib):
    assert lib.xqa_decode(None, None, 0, None, None) == X.XQA_ERR_INVALID_ARG


@pytest.mark.parametrize("buf,nbytes,sink,words", [
    (None, 1 << 20, 0x10000, 16),     # no buffer
    (0x10000, 0, 0x10000, 16),        # nothing to read
    (0x10000, 1000, 0x10000, 16),     # not a multiple of 16 bytes
    (0x10008, 1 << 20, 0x10000, 16),  # buffer not 16-byte aligned
    (0x10000, 1 << 20, None, 16),     # no sink
    (0x10000, 1 << 20, 0x10000, 0),   # no sink words
])
def test_read_probe_rejects_bad_arguments_before_launch(lib, buf, nbytes, sink, words):
    assert lib.xqa_read_bandwidth_probe(buf, nbytes, sink, words, None) == X.XQA_ERR_INVALID_ARG
    assert "read probe" in lib.xqa_last_error().decode()


def test_semaphore_count_is_one_per_row_group(lib):
    assert lib.xqa_semaphore_count(ctypes.byref(fake_params())) == 4 * 8
    # 16-bit K/V: more than 16 rows per kv head (D=128) run 128-row tensor-core tiles
    p = fake_params(num_q_heads=64, q_seq_len=8)       # 64 rows
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 1
    p = fake_params(num_q_heads=64, q_seq_len=16)      # 128 rows
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 1
    p = fake_params(num_q_heads=64, q_seq_len=32)      # 256 rows -> two row groups
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 2
    # e4m3 K/V: warp row groups of up to 64 rows
    p = fake_params(num_q_heads=64, q_seq_len=8, kv_dtype=X.XQA_E4M3)
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 1
    p = fake_params(num_q_heads=64, q_seq_len=16, kv_dtype=X.XQA_E4M3)
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 2
    # D=64: 32 rows (two blocks per warp), then 128-row tensor-core tiles
    p = fake_params(head_dim=64, num_q_heads=64, q_seq_len=4)
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 1
    p = fake_params(head_dim=64, num_q_heads=256, q_seq_len=4)
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 1
    p = fake_params(head_dim=64, num_q_heads=256, q_seq_len=8)
    assert lib.xqa_semaphore_count(ctypes.byref(p)) == 4 * 8 * 2


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_decode_20_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "xqa_oracle" not in text, f


def test_merge_params_struct_layout_matches_c(tmp_path):
    fields = [f for f, _ in X.XqaMergeParams._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "xqa.h"', "int main(void){",
            'printf("%zu\\n", sizeof(xqa_merge_params));']
    prog += [f'printf("%zu\\n", offsetof(xqa_merge_params, {f}));' for f in fields]
    prog += ["return 0;}"]
    src = tmp_path / "mlayout.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "mlayout"
    subprocess.run(["gcc", "-I" + os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(X.XqaMergeParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(X.XqaMergeParams, f).offset == off, f


def fake_merge(**over):
    """A well-formed merge parameter block with fake (never dereferenced) pointers."""
    p = X.XqaMergeParams()
    p.output = p.prefix_output = p.suffix_output = 0x10000
    p.output_lse = p.prefix_lse = p.suffix_lse = 0x20000
    p.dtype = X.XQA_BF16
    p.num_tokens, p.num_heads, p.head_dim, p.tokens_with_prefix = 4, 2, 64, 4
    p.out_stride_token = p.prefix_stride_token = p.suffix_stride_token = 128
    p.out_stride_head = p.prefix_stride_head = p.suffix_stride_head = 64
    p.lse_stride_token, p.lse_stride_head = 2, 1
    for k, v in over.items():
        setattr(p, k, v)
    return p


MERGE_BAD = [
    (dict(dtype=X.XQA_E4M3), "dtype"),
    (dict(head_dim=12), "head_dim"),
    (dict(tokens_with_prefix=5), "tokens_with_prefix"),
    (dict(prefix_output=0), "NULL"),
    (dict(suffix_output=0x10004), "aligned"),
    (dict(prefix_stride_head=60), "strides"),
    (dict(lse_stride_token=-1), "lse strides"),
]


@pytest.mark.parametrize("over,text", MERGE_BAD, ids=[t for _, t in MERGE_BAD])
def test_merge_validation_rejects_before_launch(lib, over, text):
    st = lib.xqa_merge_attn_states(ctypes.byref(fake_merge(**over)), None)
    assert st == X.XQA_ERR_INVALID_ARG
    assert text in lib.xqa_last_error().decode()


def test_merge_of_zero_tokens_is_a_no_op(lib):
    assert lib.xqa_merge_attn_states(ctypes.byref(fake_merge(num_tokens=0, tokens_with_prefix=0)),
                                     None) == X.XQA_OK


def test_misaligned_lse_rejected(lib):
    p = fake_params(lse=0x10002)
    assert lib.xqa_decode(ctypes.byref(p), None, 0, None, None) == X.XQA_ERR_INVALID_ARG
    assert "lse" in lib.xqa_last_error().decode()


def test_prep_params_struct_layout_matches_c(tmp_path):
    fields = [f for f, _ in X.XqaMlaPrepParams._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "xqa.h"', "int main(void){",
            'printf("%zu\\n", sizeof(xqa_mla_prep_params));']
    prog += [f'printf("%zu\\n", offsetof(xqa_mla_prep_params, {f}));' for f in fields]
    prog += ["return 0;}"]
    src = tmp_path / "playout.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "playout"
    subprocess.run(["gcc", "-I" + os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(X.XqaMlaPrepParams)
    for f, off in zip(fields, vals[1:]):
        assert getattr(X.XqaMlaPrepParams, f).offset == off, f


def fake_prep(**over):
    p = X.XqaMlaPrepParams()
    p.ql_nope = p.q_pe = p.kv_c = p.k_pe = p.kv_cache = p.q_out = 0x10000
    p.positions = p.slot_mapping = 0x20000
    p.cos_sin_cache = 0x30000
    p.max_position = 4096
    p.ql_stride_token, p.ql_stride_head = 128 * 512, 512
    p.qpe_stride_token, p.qpe_stride_head = 128 * 64, 64
    p.kvc_stride_token, p.kpe_stride_token = 512, 64
    p.num_slots, p.num_tokens, p.num_heads, p.kv_lora_rank, p.rope_dim = 640, 4, 128, 512, 64
    for k, v in over.items():
        setattr(p, k, v)
    return p


PREP_BAD = [
    (dict(rope_dim=60), "multiples of 8"),
    (dict(num_heads=0), "num_heads"),
    (dict(kv_cache=0), "NULL"),
    (dict(q_out=0x10008), "aligned"),
    (dict(qpe_stride_head=65), "strides"),
    (dict(cos_sin_cache=0), "cos_sin_cache"),
]


@pytest.mark.parametrize("over,text", PREP_BAD, ids=[t for _, t in PREP_BAD])
def test_prep_validation_rejects_before_launch(lib, over, text):
    assert lib.xqa_mla_decode_prep(ctypes.byref(fake_prep(**over)), None) == X.XQA_ERR_INVALID_ARG
    assert text in lib.xqa_last_error().decode()


# ---------------------------------------------------------------- MLA sizing
MLA_PARTIAL = 128 * (512 + 4) * 4  # one fp32 partial: 128 rows of 512 + (m, l) + padding


def mla_params(**over):
    base = dict(num_kv_heads=1, num_q_heads=128, head_dim=576, pages_per_seq=512, num_pages=4096)
    base.update(over)
    return fake_params(**base)


@pytest.mark.parametrize("sm,clusters", [(152, 76), (2, 1), (1000, 128)])
def test_mla_workspace_persistent_clusters(lib, sm, clusters):
    """Up to 256 sequences: one persistent cluster per SM pair (at most 128), two
    partial slots each; a single cluster needs no partials.  Two semaphores
    per sequence (its finished pieces and its finished merge items), then the
    merge kernel's item counter and its count of finished CTAs."""
    p = mla_params(batch_size=64)
    expect = clusters * 2 * MLA_PARTIAL if clusters > 1 else 0
    assert lib.xqa_mla_workspace_size(ctypes.byref(p), 512, sm) == expect
    assert lib.xqa_mla_semaphore_count(ctypes.byref(p), 512) == 64 * 2 + 2


def test_binding_refuses_short_semaphores_before_launch(lib):
    """The C ABI takes the semaphores as a bare pointer; the binding checks the
    tensor against the sizing query and raises before any launch."""
    import torch
    short = torch.zeros(64 * 2, dtype=torch.int32)  # two short of 2 B + 2
    with pytest.raises(X.XqaError) as e:
        X.xqa_mla_decode(mla_params(batch_size=64), 512, None, short)
    assert e.value.status == X.XQA_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(X.XqaError) as e:
        X.xqa_decode(fake_params(), None, torch.zeros(4 * 8 - 1, dtype=torch.int32))
    assert e.value.status == X.XQA_ERR_WORKSPACE_TOO_SMALL


def test_mla_workspace_fixed_splits_above_256_sequences(lib):
    """Above 256 sequences: a partial per (sequence, split) of a fixed page count
    aimed at 3 waves of SM pairs (at least 1024 tokens per split)."""
    p = mla_params(batch_size=300)
    assert lib.xqa_mla_workspace_size(ctypes.byref(p), 512, 152) == 0  # one split each
    # 500 pairs x 3 waves / 300 sequences -> 5 splits of 103 pages
    assert lib.xqa_mla_workspace_size(ctypes.byref(p), 512, 1000) == 300 * 5 * MLA_PARTIAL


def test_rebuild_is_keyed_on_content_not_mtime(tmp_path):
    """A library built from other sources is stale even when it is newer than
    them: the stamp beside it records the sources' digest, not a time."""
    src = tmp_path / "kernel.cu"
    src.write_text("int a = 1;\n")
    lib, stamp = tmp_path / "lib.so", tmp_path / "lib.so.sha256"
    lib.write_bytes(b"built")
    digest = B.source_digest([str(src)])
    stamp.write_text(digest + "\n")
    assert B.is_current(str(lib), str(stamp), B.source_digest([str(src)]))
    # same length, older modification time than the library: only the content moved
    st = os.stat(src)
    src.write_text("int a = 2;\n")
    os.utime(src, (st.st_atime - 100, st.st_mtime - 100))
    assert os.path.getmtime(lib) > os.path.getmtime(src)
    assert not B.is_current(str(lib), str(stamp), B.source_digest([str(src)]))
    assert not B.is_current(str(tmp_path / "missing.so"), str(stamp), digest)


def test_output_alignment_checked_before_launch(lib):
    """Four 16-bit outputs go out as one 8-byte store: an output 4 bytes off an
    8-byte boundary is rejected on the host (nothing is launched)."""
    p = fake_params(output=0x10004)
    assert lib.xqa_decode(ctypes.byref(p), None, 0, None, None) == X.XQA_ERR_INVALID_ARG
    assert "output must be 8-byte aligned" in lib.xqa_last_error().decode()
    # an e4m3 output needs 4 bytes
    # (head_dim 64 is unsupported with fp8 KV: the call fails on that later
    # check, after alignment passed, and launches nothing on any machine)
    p = fake_params(output=0x10004, kv_dtype=X.XQA_E4M3, out_dtype=X.XQA_E4M3, head_dim=64)
    assert lib.xqa_decode(ctypes.byref(p), None, 0, None, None) == X.XQA_ERR_UNSUPPORTED
    assert "head_dim" in lib.xqa_last_error().decode()
    p = fake_params(output=0x10002, kv_dtype=X.XQA_E4M3, out_dtype=X.XQA_E4M3)
    assert lib.xqa_decode(ctypes.byref(p), None, 0, None, None) == X.XQA_ERR_INVALID_ARG
    assert "4-byte aligned" in lib.xqa_last_error().decode()


@pytest.mark.parametrize("field", ["page_table", "seq_lens", "sinks", "error_word", "q_scale_dev",
                                   "kv_scale_dev"])
def test_int_and_float_pointers_need_4_byte_alignment(lib, field):
    p = fake_params(**{field: 0x10002})
    assert lib.xqa_decode(ctypes.byref(p), None, 0, None, None) == X.XQA_ERR_INVALID_ARG
    assert "4-byte aligned" in lib.xqa_last_error().decode()


def test_merge_lse_alignment_checked(lib):
    st = lib.xqa_merge_attn_states(ctypes.byref(fake_merge(suffix_lse=0x20002)), None)
    assert st == X.XQA_ERR_INVALID_ARG
    assert "lse arrays must be 4-byte aligned" in lib.xqa_last_error().decode()


def test_prep_index_alignment_checked(lib):
    assert lib.xqa_mla_decode_prep(ctypes.byref(fake_prep(slot_mapping=0x20004)), None) == X.XQA_ERR_INVALID_ARG
    assert "8-byte aligned" in lib.xqa_last_error().decode()
