"""The C ABI without a GPU: the in-tree library builds and loads, exports every
function include/*.h declares, its ctypes structs match the C layout, and the
host-only entry points behave (no compute call is made here)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def libs():
    from engram_hashed_gram_gb300 import build as B
    B.build()
    from engram_hashed_gram_gb300 import _lib
    return _lib


def declared_functions(header):
    text = open(os.path.join(INCLUDE, header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*ENGRAM(?:_SYNTH)?_API\s+(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    # every function declaration carries the export macro
    plain = re.findall(r"^(?:engram_status|void|int32_t|const char\*)\s+(engram_[a-z_]+)\s*\(", text, flags=re.M)
    assert not plain, f"declared without the export macro: {plain}"
    return sorted(set(names))


def exported(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_every_declared_function_is_exported(libs):
    for header, lib in (("engram.h", "libengram.so"), ("engram_synth.h", "libengram_synth.so")):
        names = declared_functions(header)
        assert names, header
        syms = exported(libs.lib_file(lib))
        missing = [n for n in names if n not in syms]
        assert not missing, f"{lib} lacks {missing}"
        handle = ctypes.CDLL(libs.lib_file(lib))
        for n in names:
            getattr(handle, n)


def test_bindings_cover_the_header(libs):
    assert sorted(libs.ENGRAM_FUNCS) == declared_functions("engram.h")
    assert sorted(libs.SYNTH_FUNCS) == declared_functions("engram_synth.h")


def test_struct_layout_matches_c(libs, tmp_path):
    probe = tmp_path / "probe.c"
    probe.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "engram.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f))
int main(void) {
  printf("engram_config %zu\n", sizeof(engram_config));
  F(engram_config, dim); F(engram_config, hc_mult); F(engram_config, n_cols); F(engram_config, head_dim);
  F(engram_config, scale_block); F(engram_config, scale_fmt); F(engram_config, num_rows); F(engram_config, eps);
  F(engram_config, clamp); F(engram_config, max_tokens); F(engram_config, check_ids); F(engram_config, fuse_gate);
  F(engram_config, wkv_fmt); F(engram_config, row_offset);
  printf("engram_weights %zu\n", sizeof(engram_weights));
  F(engram_weights, table); F(engram_weights, scale); F(engram_weights, wkv); F(engram_weights, q_weight);
  F(engram_weights, k_weight); F(engram_weights, wkv_scale);
  printf("engram_plan_info %zu\n", sizeof(engram_plan_info));
  F(engram_plan_info, splits); F(engram_plan_info, ctas); F(engram_plan_info, cta_pairs);
  F(engram_plan_info, rem_tiles); F(engram_plan_info, rem_splits); F(engram_plan_info, fused_gate);
  printf("engram_hash_config %zu\n", sizeof(engram_hash_config));
  F(engram_hash_config, n_layers); F(engram_hash_config, max_ngram_size); F(engram_hash_config, n_heads);
  F(engram_hash_config, max_batch); F(engram_hash_config, max_len); F(engram_hash_config, vocab_size);
  F(engram_hash_config, pad_id); F(engram_hash_config, dead_id);
  return 0;
}
''')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(probe), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    c = dict(l.rsplit(" ", 1) for l in lines if l)
    assert int(c["engram_config"]) == ctypes.sizeof(libs.EngramConfig)
    assert int(c["engram_weights"]) == ctypes.sizeof(libs.EngramWeights)
    assert int(c["engram_hash_config"]) == ctypes.sizeof(libs.EngramHashConfig)
    assert int(c["engram_plan_info"]) == ctypes.sizeof(libs.EngramPlanInfo)
    names = {libs.EngramConfig: "engram_config", libs.EngramWeights: "engram_weights",
             libs.EngramHashConfig: "engram_hash_config", libs.EngramPlanInfo: "engram_plan_info"}
    for T, cname in names.items():
        for f, _ in T._fields_:
            assert int(c[f"{cname}.{f}"]) == getattr(T, f).offset, f


def test_host_only_entry_points(libs):
    lib = libs.engram()
    assert lib.engram_abi_version() == 105
    for code, text in ((0, b"ok"), (-1, b"invalid argument"), (-4, b"hash id outside the table"),
                       (-5, b"kernel wait timed out"), (-6, b"unsupported shape or format"), (7, b"unknown status")):
        assert lib.engram_status_string(code) == text
    # null arguments are refused before any CUDA call
    assert lib.engram_create(None, None, None) == -1
    h = ctypes.c_void_p()
    cfg = libs.EngramConfig(dim=5120, hc_mult=4, n_cols=24, head_dim=256, scale_block=128, num_rows=10,
                            eps=1e-6, clamp=1e-6, max_tokens=8)
    w = libs.EngramWeights()
    assert lib.engram_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w)) == -1
    assert lib.engram_forward(None, None, None, None, None, 1, 1, None) == -1
    assert lib.engram_lookup_project(None, None, None, 1, 1, None) == -1
    assert lib.engram_gate_apply(None, None, None, None, None, None, 1, 1, None) == -1
    assert lib.engram_lookup(None, None, None, 1, 1, None) == -1
    assert lib.engram_forward_rows(None, None, None, None, None, 1, 1, None) == -1
    assert lib.engram_sync_status(None, None, None) == -1
    assert lib.engram_plan(None, 1, None, None) == -1
    assert lib.engram_describe_plan(None, 1, None) == -1
    assert lib.engram_set_sm_budget(None, 8) == -1
    assert lib.engram_test_hook(None, 1) == -1
    assert lib.engram_enable_stage_timing(None, 1) == -1
    assert lib.engram_stage_times(None, None) == -1
    assert lib.engram_stage_times_n(None, 1, None) == -1
    assert lib.engram_hash(None, None, None, None, None, None, None, None, 0, None, 1, 1, None) == -1
    # more primes than the kernel's shared-memory table holds, refused before any CUDA call
    hc = libs.EngramHashConfig(n_layers=97, max_ngram_size=3, n_heads=32, max_batch=1, max_len=1, vocab_size=1,
                               pad_id=2, dead_id=-1)
    assert lib.engram_hash(ctypes.byref(hc), None, None, None, None, None, None, None, 0, None, 0, 0, None) == -6
    hc.n_layers = 96                                        # 96 * 2 * 32 = 6144 primes: accepted, empty batch
    assert lib.engram_hash(ctypes.byref(hc), None, None, None, None, None, None, None, 0, None, 0, 0, None) == 0
    lib.engram_destroy(None)
    syn = libs.synth()
    assert syn.engram_synth_fill_table(None, None, 0, 1, 256, 128, 0, 0, None, None, None) == -1


def test_product_path_does_not_import_the_oracle():
    """The package never imports oracle/: load it in a fresh interpreter and
    check sys.modules."""
    code = ("import sys; import engram_hashed_gram_gb300.layer, engram_hashed_gram_gb300.synth_device; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, check=True)
    assert r.stdout.strip() == "False"
    pkg = os.path.join(ROOT, "engram_hashed_gram_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_binding_refuses_a_host_table_the_device_cannot_read():
    """EngramLayer takes a CUDA table or a pinned host table; an ordinary
    (pageable) host tensor is refused before anything reaches the library."""
    import torch
    from engram_hashed_gram_gb300.layer import EngramLayer
    table = torch.zeros((4, 256), dtype=torch.uint8)
    assert not table.is_pinned()
    with pytest.raises(ValueError, match="pinned"):
        EngramLayer(table, torch.zeros((4, 2)), torch.zeros(1), torch.zeros(1), torch.zeros(1))
