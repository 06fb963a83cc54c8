"""The C ABI from plain C99: include/kvx.h compiles as C with warnings as errors, a C
program links against libkvx.so, and the host-only entry points it calls agree with the
Python binding and with closed forms.  No GPU needed."""
import ctypes
import os
import shutil
import subprocess

import pytest

from paged_kv_gather_gb300 import kvx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def abi_values(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = kvx.library_path()
    exe = str(tmp_path_factory.mktemp("abi") / "abi_check")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", exe,
                    "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return dict(line.split(" ", 1) for line in out.strip().splitlines())


def test_struct_sizes_match_the_binding(abi_values):
    assert int(abi_values["sizeof_pool"]) == ctypes.sizeof(kvx.kvx_pool)
    assert int(abi_values["sizeof_request"]) == kvx.REQUEST_DTYPE.itemsize
    assert int(abi_values["sizeof_chunk"]) == kvx.CHUNK_DTYPE.itemsize
    assert int(abi_values["sizeof_cfg"]) == ctypes.sizeof(kvx.kvx_launch_cfg)
    assert int(abi_values["sizeof_link_model"]) == ctypes.sizeof(kvx.kvx_link_model)
    assert int(abi_values["version"]) == kvx.kvx_version()


def test_field_offsets_match_the_binding(abi_values):
    """Every field of every ABI struct sits where the binding puts it (sizes alone would not
    catch two swapped fields of the same size)."""
    offs = {k[len("off_"):]: int(v) for k, v in abi_values.items() if k.startswith("off_")}
    for struct in (kvx.kvx_pool, kvx.kvx_launch_cfg, kvx.kvx_link_model):
        for name, _ in struct._fields_:
            assert offs.pop(f"{struct.__name__}_{name}") == getattr(struct, name).offset, name
    for cname, dtype in (("kvx_request", kvx.REQUEST_DTYPE), ("kvx_chunk", kvx.CHUNK_DTYPE)):
        for name in dtype.names:
            assert offs.pop(f"{cname}_{name}") == dtype.fields[name][1], name
    assert not offs, f"fields the binding does not have: {sorted(offs)}"


def test_host_entry_points_from_c(abi_values):
    assert int(abi_values["validate_ok"]) == kvx.KVX_OK
    assert int(abi_values["validate_misaligned"]) == kvx.KVX_ERR_ALIGNMENT
    assert int(abi_values["validate_tokens"]) != kvx.KVX_OK
    # Segments: chunk 0 covers pages 0..15 (16 pages) x 4 layers x K/V; chunk 1 tokens
    # 256..555 cover pages 16..34 (19 pages) x 8; chunk 2 tokens 556..999 cover pages
    # 34..62 (29 pages) x 2 layers x 2.
    assert int(abi_values["segments"]) == 16 * 8 + 19 * 8 + 29 * 4
    assert int(abi_values["bytes"]) == (256 * 8 + 300 * 8 + 444 * 4) * 2048
    # Window [1, 3): two layers of every chunk (chunk 2 holds layers 1..2).
    assert int(abi_values["segments_window"]) == 16 * 4 + 19 * 4 + 29 * 4
    assert int(abi_values["bytes_window"]) == (256 + 300 + 444) * 4 * 2048
    # Policy: whole pages, within the default target, per-layer when streaming.
    t, lay = int(abi_values["policy_tokens"]), int(abi_values["policy_layers"])
    assert t % 16 == 0 and lay == 4 and t * lay * 2 * 2048 <= 2 << 20
    ts, ls = int(abi_values["policy_stream_tokens"]), int(abi_values["policy_stream_layers"])
    assert ts % 16 == 0 and ls == 1 and ts * 2 * 2048 <= 1 << 20
    m = kvx.kvx_default_link_model()
    assert float(abi_values["estimate_load_us"]) == pytest.approx(
        kvx.kvx_estimate_us(m, kvx.KVX_OP_LOAD, 1 << 32), rel=1e-9)
    assert float(abi_values["estimate_roundtrip_us"]) == pytest.approx(
        kvx.kvx_estimate_pair_us(m, kvx.KVX_OP_ROUNDTRIP, 1 << 32, 1 << 32, 32768), rel=1e-9)
    assert abi_values["status_string_overlap"] == kvx.kvx_status_string(kvx.KVX_ERR_OVERLAP)
