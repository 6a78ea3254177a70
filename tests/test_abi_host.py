"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, its structs match the header, and configuration validation behaves.
No GPU is touched (no compute call is made)."""

import ctypes
import os
import re

import pytest

from decoder_only_forward_gb300 import build as dec_build
from decoder_only_forward_gb300 import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dec.h")


@pytest.fixture(scope="module")
def dec():
    dec_build.build()
    from decoder_only_forward_gb300 import dec as d
    return d


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z0-9_]+)\s*\(", text)))


def test_header_functions_all_exported(dec):
    declared = _declared_functions()
    assert len(declared) >= 15
    lib = ctypes.CDLL(dec._LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in dec.h but not exported"
    assert sorted(dec.EXPORTED) == declared


def test_config_struct_matches_header(dec):
    text = open(HEADER).read()
    body = re.search(r"typedef struct dec_config \{(.*?)\} dec_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b(int32_t|float)\s+([a-z_0-9]+)\s*;", body)
    assert [n for _, n in fields] == [n for n, _ in dec.Config._fields_]
    for (ty, n), (cn, ct) in zip(fields, dec.Config._fields_):
        assert (ct is ctypes.c_float) == (ty == "float"), n
    assert ctypes.sizeof(dec.Config) == 4 * len(fields)


@pytest.mark.parametrize("name", sorted(synthetic.WORKLOADS))
def test_workloads_validate(dec, name):
    w = synthetic.workload(name)
    for kv in ("f32", "bf16"):
        c = dec.make_config(w, kv)
        st, msg = dec.validate(c)
        assert st == dec.DEC_OK, msg
        assert dec.workspace_bytes(c) > 0


def test_workspace_covers_kv_cache(dec):
    w = synthetic.workload("mistral-7b")
    c32, c16 = dec.make_config(w, "f32"), dec.make_config(w, "bf16")
    kv32 = 2 * w["n_layers"] * w["max_seq"] * w["n_kv_heads"] * w["head_dim"] * 4
    assert dec.workspace_bytes(c32) >= kv32
    assert dec.workspace_bytes(c32) - dec.workspace_bytes(c16) >= kv32 // 2


@pytest.mark.parametrize("field,value,needle", [
    ("n_layers", 0, "positive"),
    ("n_kv_heads", 3, "multiple"),
    ("head_dim", 15, "even"),
    ("rms_eps", 0.0, "positive"),
    ("rope_theta", -1.0, "positive"),
    ("n_experts_used", 1, "dense"),
    ("weight_dtype", 7, "weight_dtype"),
    ("sliding_window", 16, "window"),
])
def test_invalid_configs_rejected(dec, field, value, needle):
    c = dec.make_config(synthetic.workload("toy"))
    setattr(c, field, value)
    st, msg = dec.validate(c)
    assert st == dec.DEC_EINVAL
    assert needle in msg
    assert dec.workspace_bytes(c) == 0


def test_expert_count_rules(dec):
    w = synthetic.workload("mixtral-8x7b")
    c = dec.make_config(w)
    c.n_experts_used = 9
    assert dec.validate(c)[0] == dec.DEC_EINVAL
    c.n_experts_used = 0
    assert dec.validate(c)[0] == dec.DEC_EINVAL
    c.n_experts_used = 2
    assert dec.validate(c)[0] == dec.DEC_OK


def test_llama3_fields_checked(dec):
    c = dec.make_config(synthetic.workload("toy"))
    c.rope_llama3 = 1
    assert dec.validate(c)[0] == dec.DEC_EINVAL
    c.rope_factor, c.rope_low_freq_factor, c.rope_high_freq_factor, c.rope_orig_ctx = 8.0, 1.0, 4.0, 8192
    assert dec.validate(c)[0] == dec.DEC_OK


def test_create_rejects_bad_arguments_without_gpu(dec):
    # Argument errors are detected before any CUDA call: NULL weights / workspace.
    c = dec.make_config(synthetic.workload("toy"))
    h = ctypes.c_void_p()
    st = dec.lib.dec_create(ctypes.byref(c), None, None, 0, None, ctypes.byref(h))
    assert st == dec.DEC_EINVAL and not h.value
    assert b"weights" in dec.lib.dec_last_error(None)


def test_workspace_grows_by_one_kv_ring_set_per_sequence(dec):
    w = synthetic.workload("mistral-7b")
    base = dec.workspace_bytes(dec.make_config(w, "f32"))
    rows = (w["max_seq"] + 63) // 64 * 64
    ring_set = 2 * w["n_layers"] * rows * w["n_kv_heads"] * w["head_dim"] * 4
    for n in (2, 5):
        assert dec.workspace_bytes(dec.make_config(w, "f32", n_seqs=n)) - base == (n - 1) * ring_set
    assert dec.workspace_bytes(dec.make_config(w, "f32", n_seqs=1)) == base


def test_n_seqs_checked(dec):
    c = dec.make_config(synthetic.workload("toy"))
    c.n_seqs = -1
    st, msg = dec.validate(c)
    assert st == dec.DEC_EINVAL and "n_seqs" in msg
    c.n_seqs = 8
    assert dec.validate(c)[0] == dec.DEC_OK


def test_norm_variant_fields_checked(dec):
    c = dec.make_config(synthetic.workload("toy", qk_norm="head", sandwich_norms=True))
    assert (c.qk_norm, c.sandwich_norms) == (1, 1)
    assert dec.validate(c)[0] == dec.DEC_OK
    c.kv_dtype = dec.DEC_BF16
    st, msg = dec.validate(c)
    assert st == dec.DEC_EINVAL and "qk_norm" in msg
    c.kv_dtype, c.qk_norm = dec.DEC_F32, 3
    assert dec.validate(c)[0] == dec.DEC_EINVAL
    c.qk_norm, c.sandwich_norms = 2, 2
    assert dec.validate(c)[0] == dec.DEC_EINVAL


def test_paged_cache_config_and_arena_size(dec):
    w = synthetic.workload("mistral-7b")
    c = dec.make_config(w, "f32", n_seqs=64, page_size=16, n_pages=1024)
    assert dec.validate(c)[0] == dec.DEC_OK
    rb = w["n_kv_heads"] * w["head_dim"] * 4
    arena = 1024 * 2 * w["n_layers"] * 16 * rb
    rings = 64 * 2 * w["n_layers"] * w["max_seq"] * rb
    # The arena replaces the per-sequence rings: 1024 pages of 16 positions instead of 64 x 4096.
    flat = dec.workspace_bytes(dec.make_config(w, "f32", n_seqs=64))
    assert dec.workspace_bytes(c) - (flat - rings) - arena < 64 * 256 * 4 * 2 + 4096
    for ps, n_pages in ((8, 4), (24, 4), (16, 0)):
        bad = dec.make_config(w, "f32", page_size=ps, n_pages=n_pages)
        st, msg = dec.validate(bad)
        assert st == dec.DEC_EINVAL and ("page" in msg)


def test_weight_structs_match_header(dec):
    text = open(HEADER).read()
    body = re.search(r"typedef struct dec_layer_weights \{(.*?)\} dec_layer_weights;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"\*\s*([a-z_0-9]+)", body)
    assert names == [n for n, _ in dec.LayerWeights._fields_]
    assert ctypes.sizeof(dec.LayerWeights) == 8 * len(names)
    body = re.search(r"typedef struct dec_weights \{(.*?)\} dec_weights;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"\*\s*([a-z_0-9]+)\s*;", body)
    assert names == [n for n, _ in dec.Weights._fields_]


def test_header_is_plain_c(tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "dec.h"\nint main(void) { dec_config c = {0}; return (int)dec_workspace_bytes(&c); }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_workspace_holds_the_transposed_down_copy_when_the_ffn_fuses(dec):
    # bf16 weights, hidden a multiple of 128 and ffn a multiple of 16: the workspace
    # gains a transposed copy of every down projection (2 bytes per element) and
    # 256 x hidden floats of partial sums.  With ffn 8 past a multiple of 16 it does not
    # (its other regions grow by a little for the 8 extra columns).
    base = synthetic.workload("mistral-7b", n_layers=2, max_seq=64)
    odd = dict(base, ffn=base["ffn"] + 8)
    ws = dec.workspace_bytes(dec.make_config(base))
    ws_odd = dec.workspace_bytes(dec.make_config(odd))
    extra = 2 * base["n_layers"] * base["ffn"] * base["hidden"] + 256 * base["hidden"] * 4
    assert extra - (1 << 20) <= ws - ws_odd <= extra


def test_workspace_holds_the_current_kv_rows_for_int8_and_qk_norm_decode(dec):
    # Persistent decode with an int8 cache (head_dim 128) or the per-head QK-norm keeps the
    # new position's K and V in f32 (2 x n_kv x head_dim floats) beside the rings.
    w = synthetic.workload("mistral-7b", n_layers=2, max_seq=64)
    kd = w["n_kv_heads"] * w["head_dim"]
    f32 = dec.workspace_bytes(dec.make_config(w))
    qkn = dec.workspace_bytes(dec.make_config(dict(w, qk_norm="head")))
    assert qkn - f32 >= 2 * kd * 4 - 256   # (an empty region still takes one 256-byte slot)
