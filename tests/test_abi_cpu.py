"""CPU checks of the boundary: the library loads, exports every symbol the
header declares, agrees with the header's struct layout, and validates
configurations on the host (no GPU needed)."""
import ctypes as C
import os
import re
import subprocess

import pytest

import trainable_sparse_attention_decode_gb300 as nosa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nosa.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nosa_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 13
    lib = C.CDLL(nosa.lib_path)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_struct_layout_matches_header(tmp_path):
    # every field of both host structs, at the offset the C compiler gives it
    structs = [("nosa_config", nosa.NosaConfig), ("nosa_stats_t", nosa.NosaStats)]
    lines = []
    for cname, py in structs:
        lines.append(f'  printf("%zu\\n", sizeof({cname}));')
        lines += [f'  printf("%zu\\n", offsetof({cname}, {f}));' for f, _ in py._fields_]
    prog = tmp_path / "layout.c"
    prog.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"nosa.h\"\n"
                    "int main(void) {\n" + "\n".join(lines) + "\n  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(prog), "-o",
                    str(exe)], check=True)
    vals = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                        check=True).stdout.split()))
    want = []
    for _, py in structs:
        want.append(C.sizeof(py))
        want += [getattr(py, f).offset for f, _ in py._fields_]
    assert vals == want


def _cfg(**kw):
    base = dict(batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, dtype="bf16", k=8, k_e=6,
                max_context=4096)
    base.update(kw)
    return nosa.nosa_config(**base)


@pytest.mark.parametrize("kw,status", [
    ({}, 0),
    ({"dtype": "f32", "head_dim": 64}, 0),
    ({"k_e": 9}, 1),
    ({"k": 0, "k_e": 0}, 1),
    ({"n_q_heads": 7}, 1),
    ({"n_q_heads": 10}, 7),          # G = 5 is not compiled
    ({"head_dim": 96}, 7),
    ({"block": 32}, 7),
    ({"block": 64, "sub_block": 24}, 1),
    ({"max_context": 0}, 1),
    ({"max_context": 64 * 32768 + 1}, 7),
    ({"k": 257, "k_e": 0}, 7),
    ({"flags": 4}, 1),                # unknown flag bit
    ({"flags": 3}, 0),                # timing + bf16 pooled keys
])
def test_config_validation(kw, status):
    st, msg = nosa.nosa_config_validate(_cfg(**kw))
    assert st == status, msg
    assert (st == 0) == (msg == "")


def test_payload_bytes():
    assert nosa.nosa_payload_bytes(_cfg()) == 33024
    assert nosa.nosa_payload_bytes(_cfg(dtype="f32", head_dim=64)) == 33024
    assert nosa.nosa_payload_bytes(_cfg(head_dim=64)) == 16640
    assert nosa.nosa_payload_bytes(_cfg(dtype="f32", head_dim=128)) == 65792
    assert nosa.nosa_payload_bytes(_cfg(k_e=99)) == 0


def test_create_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(nosa.NosaError) as ei:
        nosa.nosa_create(_cfg())
    assert ei.value.status == 5 and nosa.nosa_last_error() != ""


def test_workspace_query_rejects_bad_config():
    assert nosa.nosa_attention_workspace_bytes(_cfg(k_e=99), 8) == 0


def test_frontend_rows():
    cfg = nosa.nosa_config(32, 32, 8, 128, "bf16", 64, 48, 70000)
    assert nosa.nosa_frontend_rows(cfg) == (32 + 16) * 128 + 8
    bad = nosa.nosa_config(32, 30, 8, 128, "bf16", 64, 48, 70000)
    assert nosa.nosa_frontend_rows(bad) == 0


def test_prefill_timing_without_a_timed_forward():
    # the timing query of the training-time forward needs a timed call on the
    # same thread first: STATE, no device access
    import threading
    out = {}

    def probe():
        f, a = C.c_float(1.0), C.c_float(1.0)
        out["st"] = nosa.lib.nosa_prefill_timing(C.byref(f), C.byref(a))
        out["vals"] = (f.value, a.value)

    t = threading.Thread(target=probe)
    t.start()
    t.join()
    assert out["st"] == 6  # STATE
    assert out["vals"] == (1.0, 1.0)  # outputs untouched


# --------------------------------------------------------------------------
# NUMA placement of the pinned host store: the pure rule, on fake topologies
# --------------------------------------------------------------------------
@pytest.mark.parametrize("gpu_node,mem_nodes,allowed,want", [
    (1, [0, 1], [0, 1], 1),          # two Grace dies: the GPU's own node
    (0, [0, 1], [0, 1], 0),
    (3, [0, 1, 2, 3], [0, 1, 2, 3], 3),  # four sockets
    (1, [0, 1], [0], -1),            # the GPU's node is not allowed to this process
    (2, [0, 1], [0, 1, 2], -1),      # the GPU's node has no CPUs with memory (a GPU-memory node)
    (0, [0], [0], -1),               # one memory node: nothing to choose
    (-1, [0, 1], [0, 1], -1),        # node unknown (sysfs reports -1)
    (1, [], [0, 1], -1),
])
def test_numa_placement_rule(gpu_node, mem_nodes, allowed, want):
    assert nosa.nosa_numa_choose(gpu_node, mem_nodes, allowed) == want


def test_numa_rule_null_arrays():
    assert nosa.lib.nosa_numa_choose(1, None, 2, None, 2) == -1
