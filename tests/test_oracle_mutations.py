"""The oracle's pins must fail on plausible mistakes planted in the oracle.

Each case compiles a copy of oracle/kv_oracle.c with one edit (a transposed axis, a dropped
term, a wrong index) into a temporary library, points the oracle's Python face at it, and
checks that at least one pin of tests/test_oracle_pins.py fails.  All on the CPU.
"""
import ctypes
import os
import subprocess
import sys

import pytest

import oracle.kv_oracle as ko
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(ko.__file__), "kv_oracle.c")

MUTATIONS = {
    "layer_major_kv_layer_swapped": ("index = (lr * KV + kv) * c->n_tokens + tr;",
                                     "index = (kv * c->n_layers + lr) * c->n_tokens + tr;"),
    "token_major_axes_swapped": ("index = (tr * c->n_layers + lr) * KV + kv;",
                                 "index = (lr * c->n_tokens + tr) * KV + kv;"),
    "token_in_page_dropped": ("int64_t slot = page * pool->page_size + (t % pool->page_size);",
                              "int64_t slot = page * pool->page_size;"),
    "page_table_skipped": ("int64_t page = req->page_table[t / pool->page_size];",
                           "int64_t page = t / pool->page_size;"),
    "pool_index_transposed": ("pool->pools[(int64_t)kv * pool->num_layers + layer]",
                              "pool->pools[(int64_t)layer * pool->kv_factor + kv]"),
    "chunk_layer_not_relative": ("int64_t lr = layer - c->layer_begin;",
                                 "int64_t lr = layer;"),
    "window_ignored": ("int32_t l_lo = c->layer_begin > layer_begin ? c->layer_begin : layer_begin;",
                       "int32_t l_lo = c->layer_begin;"),
    "token_offset_sign": ("int64_t tr = t - c->token_begin;", "int64_t tr = c->token_begin - t + c->n_tokens - 1;"),
    "stripe_not_padded": ("int64_t stride = (object_bytes + ORA_STRIPE_ALIGN - 1) / ORA_STRIPE_ALIGN * ORA_STRIPE_ALIGN;",
                          "int64_t stride = object_bytes;"),
}

PIN_CASES = [
    lambda: pins.test_bruteforce_every_cut_and_layer_window(2, 16),
    lambda: pins.test_bruteforce_random_multi_request_mixes(),
    lambda: pins.test_numpy_fancy_indexing_cross_check(0),
    lambda: pins.test_strata_worked_example_golden(),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation {name} does not apply"
    mutated = src.replace(old, new, 1)
    cpath = tmp_path / f"{name}.c"
    cpath.write_text(mutated)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(cpath)],
                   check=True)
    return str(lib)


def _child(path: str) -> int:
    """Run the pins against the library at ``path``; 3 = a pin failed, 0 = none did."""
    lib = ctypes.CDLL(path)
    for fn_name in ("ora_store", "ora_load"):
        fn = getattr(lib, fn_name)
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.POINTER(ko._Pool), ctypes.POINTER(ko._Request), ctypes.c_int,
                       ctypes.POINTER(ko._Chunk), ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.ora_bytes.restype = ctypes.c_int64
    lib.ora_bytes.argtypes = [ctypes.POINTER(ko._Pool), ctypes.POINTER(ko._Chunk),
                              ctypes.c_int, ctypes.c_int, ctypes.c_int]
    ko._lib_handle = lib
    for case in PIN_CASES:
        try:
            case()
        except (AssertionError, ValueError):
            return 3
    return 0


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    """A mutant either fails a pin (exit 3) or crashes on an out-of-bounds access the
    canary-padded buffers expose; it must never pass every pin (exit 0)."""
    old, new = MUTATIONS[name]
    path = _build_mutant(tmp_path, name, old, new)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (f"import sys; sys.path.insert(0, {root!r}); "
            f"from tests import test_oracle_mutations as m; sys.exit(m._child({path!r}))")
    rc = subprocess.run([sys.executable, "-c", code], capture_output=True, timeout=600).returncode
    assert rc != 0, f"no pin caught mutation {name}"
    assert rc == 3 or rc < 0, f"mutant {name} exited with unexpected code {rc}"
