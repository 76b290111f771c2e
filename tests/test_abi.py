"""The C ABI library loads, exports every entry point include/kamera.h
declares, its structs match the binding's, and host-side validation rejects
bad arguments with the documented status codes (CPU only: every call here
returns before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

import position_invariant_kv_kamera_gb300 as pk
from position_invariant_kv_kamera_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "kamera.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pk.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(kamera_\w+)\s*\(", src, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kamera_reuse_batched", "kamera_relocate", "kamera_apply_patch"):
        assert n in names
    assert set(names) == set(pk.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True).stdout
    for name in declared_functions():
        assert re.search(r"\bT " + name + r"\b", out), name


def test_abi_version_and_status_strings(lib):
    assert pk.abi_version() == 4
    assert pk.status_string(pk.KAMERA_OK) == "KAMERA_OK"
    assert pk.status_string(pk.KAMERA_ERR_CUDA) == "KAMERA_ERR_CUDA"
    assert pk.status_string(99) == "KAMERA_ERR_UNKNOWN"


def test_struct_layouts_match_header(tmp_path):
    prog = tmp_path / "sizes.c"
    prog.write_text(r'''
#include <stdio.h>
#include <stddef.h>
#include "kamera.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(kamera_model_desc), sizeof(kamera_chunk_store),
         sizeof(kamera_patch_store), sizeof(kamera_paged_pool), sizeof(kamera_reuse_item), sizeof(kamera_factor_desc));
  printf("%zu %zu %zu %zu %zu\n", offsetof(kamera_model_desc, rope_base), offsetof(kamera_reuse_item, delta),
         offsetof(kamera_reuse_item, dst_pos), offsetof(kamera_paged_pool, block_table),
         offsetof(kamera_model_desc, section_delta));
  printf("%zu %zu %zu\n", sizeof(kamera_compressed_store), offsetof(kamera_compressed_store, n_chunks),
         offsetof(kamera_compressed_store, n_rows));
  return 0;
}
''')
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-I" + _build.INCLUDE, "-o", str(exe), str(prog)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    sizes = [int(x) for x in lines[0].split()]
    assert sizes == [ctypes.sizeof(pk.kamera_model_desc), ctypes.sizeof(pk.kamera_chunk_store),
                     ctypes.sizeof(pk.kamera_patch_store), ctypes.sizeof(pk.kamera_paged_pool),
                     pk.REUSE_ITEM.itemsize, ctypes.sizeof(pk.kamera_factor_desc)]
    offs = [int(x) for x in lines[1].split()]
    assert offs == [pk.kamera_model_desc.rope_base.offset, pk.REUSE_ITEM.fields["delta"][1],
                    pk.REUSE_ITEM.fields["dst_pos"][1], pk.kamera_paged_pool.block_table.offset,
                    pk.kamera_model_desc.section_delta.offset]
    comp = [int(x) for x in lines[2].split()]
    assert comp == [ctypes.sizeof(pk.kamera_compressed_store), pk.kamera_compressed_store.n_chunks.offset,
                    pk.kamera_compressed_store.n_rows.offset]


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _gqa_model(**kw):
    m = pk.model_desc(pk.KAMERA_GQA, 2, 4, 128, rope_base=1e6)
    for k, v in kw.items():
        setattr(m, k, v)
    return m


def _pool(**kw):
    p = pk.kamera_paged_pool(FAKE, FAKE + 4096, 16, 64, FAKE + 8192, 1, 16)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _store():
    return pk.kamera_chunk_store(FAKE, 1 << 20, FAKE, FAKE, 4)


def _reuse(model, pool, store=None, patches=None, n=1):
    st = store if store is not None else _store()
    return pk.kamera_reuse_batched(model, st, patches, FAKE, n, pool, None, None, raise_on_error=False)


def test_validation_null_pointers(lib):
    assert pk.kamera_reuse_batched(None, _store(), None, FAKE, 1, _pool(), None, None, False) == pk.KAMERA_ERR_NULL
    assert pk.kamera_reuse_batched(_gqa_model(), _store(), None, FAKE, 1, None, None, None, False) == pk.KAMERA_ERR_NULL
    assert pk.kamera_reuse_batched(_gqa_model(), None, None, FAKE, 1, _pool(), None, None, False) == pk.KAMERA_ERR_NULL
    assert pk.kamera_reuse_batched(_gqa_model(), _store(), None, None, 1, _pool(), None, None, False) == pk.KAMERA_ERR_NULL
    assert _reuse(_gqa_model(), _pool(k=None)) == pk.KAMERA_ERR_NULL
    assert _reuse(_gqa_model(), _pool(v=None)) == pk.KAMERA_ERR_NULL
    assert _reuse(_gqa_model(), _pool(block_table=None)) == pk.KAMERA_ERR_NULL
    assert pk.kamera_apply_patch(_gqa_model(), None, FAKE, 1, _pool(), None, None, False) == pk.KAMERA_ERR_NULL
    assert "NULL" in pk.last_error()


def test_validation_invalid_arguments(lib):
    assert _reuse(_gqa_model(family=7), _pool()) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(num_layers=0), _pool()) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(pairing=3), _pool()) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(patch_frame=2), _pool()) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(num_kv_heads=0), _pool()) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(), _pool(page_size=48)) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(), _pool(page_size=4)) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(), _pool(num_pages=0)) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse(_gqa_model(), _pool(), n=-1) == pk.KAMERA_ERR_INVALID_ARG
    patches = pk.kamera_patch_store(FAKE, 1 << 20, FAKE, FAKE, 4, 12)
    assert _reuse(_gqa_model(), _pool(), patches=patches) == pk.KAMERA_ERR_INVALID_ARG
    mla = pk.model_desc(pk.KAMERA_MLA, 2, rope_dim=64, latent_dim=512)
    assert _reuse(mla, _pool()) == pk.KAMERA_ERR_INVALID_ARG  # MLA pools carry no V
    bad_base = _gqa_model(rope_base=-1.0)
    assert _reuse(bad_base, _pool()) == pk.KAMERA_ERR_INVALID_ARG
    m = _gqa_model()
    m.rope_sections[0], m.rope_sections[1], m.rope_sections[2] = 16, 24, 23  # must sum to rope_dim/2 = 64
    assert _reuse(m, _pool()) == pk.KAMERA_ERR_INVALID_ARG
    m.rope_sections[2] = -1
    assert _reuse(m, _pool()) == pk.KAMERA_ERR_INVALID_ARG


def test_validation_unsupported_shapes(lib):
    assert _reuse(_gqa_model(head_dim=80), _pool()) == pk.KAMERA_ERR_UNSUPPORTED
    assert _reuse(_gqa_model(head_dim=512), _pool()) == pk.KAMERA_ERR_UNSUPPORTED
    assert _reuse(_gqa_model(rope_dim=96), _pool()) == pk.KAMERA_ERR_UNSUPPORTED
    assert _reuse(_gqa_model(num_kv_heads=32), _pool()) == pk.KAMERA_ERR_UNSUPPORTED  # D = 4096
    mla = pk.model_desc(pk.KAMERA_MLA, 2, rope_dim=64, latent_dim=500)
    assert _reuse(mla, _pool(v=None)) == pk.KAMERA_ERR_UNSUPPORTED
    huge = _pool(num_pages=1 << 26)
    assert _reuse(_gqa_model(), huge) == pk.KAMERA_ERR_UNSUPPORTED  # > 2^31 pool rows


def test_validation_alignment(lib):
    assert _reuse(_gqa_model(), _pool(k=FAKE + 8)) == pk.KAMERA_ERR_ALIGNMENT
    st = pk.kamera_chunk_store(FAKE + 2, 1 << 20, FAKE, FAKE, 4)
    assert _reuse(_gqa_model(), _pool(), store=st) == pk.KAMERA_ERR_ALIGNMENT
    assert pk.kamera_reuse_batched(_gqa_model(), _store(), None, FAKE, 1, _pool(), FAKE + 2, None,
                                   False) == pk.KAMERA_ERR_ALIGNMENT


def test_empty_batch_is_a_no_op(lib):
    assert _reuse(_gqa_model(), _pool(), n=0) == pk.KAMERA_OK


def test_factor_validation(lib):
    d = pk.kamera_factor_desc(FAKE, 300 * 256, 4, 300, 256, 16, 16, 1, FAKE)
    out = ctypes.c_size_t(0)
    assert lib.kamera_factor_workspace_size(None, ctypes.byref(out)) == pk.KAMERA_ERR_NULL
    bad = pk.kamera_factor_desc(FAKE, 300 * 256, 4, 300, 256, 12, 16, 1, FAKE)
    assert lib.kamera_factor_workspace_size(ctypes.byref(bad), ctypes.byref(out)) == pk.KAMERA_ERR_INVALID_ARG
    bad = pk.kamera_factor_desc(FAKE, 300 * 256, 4, 300, 256, 64, 40, 1, FAKE)  # k = 104 > 96
    assert lib.kamera_factor_workspace_size(ctypes.byref(bad), ctypes.byref(out)) == pk.KAMERA_ERR_INVALID_ARG
    bad = pk.kamera_factor_desc(FAKE, 300 * 256, 4, 300, 4096, 16, 16, 1, FAKE)
    assert lib.kamera_factor_workspace_size(ctypes.byref(bad), ctypes.byref(out)) == pk.KAMERA_ERR_UNSUPPORTED
    bad = pk.kamera_factor_desc(FAKE, 100, 4, 300, 256, 16, 16, 1, FAKE)  # stride < T*D
    assert lib.kamera_factor_workspace_size(ctypes.byref(bad), ctypes.byref(out)) == pk.KAMERA_ERR_INVALID_ARG
    assert pk.kamera_factor_patches(d, None, FAKE, 1 << 20, FAKE, 1 << 30, None, False) == pk.KAMERA_ERR_NULL
    assert pk.kamera_factor_patches(d, FAKE, FAKE, 1 << 20, FAKE + 16, 1 << 30, None, False) == pk.KAMERA_ERR_ALIGNMENT
    empty = pk.kamera_factor_desc(None, 0, 0, 300, 256, 16, 16, 1, None)
    assert pk.kamera_factor_patches(empty, None, None, 0, None, 0, None, False) == pk.KAMERA_OK


def test_launch_tuning_set_get_and_validation(lib):
    """The process-wide launch tuning round-trips, rejects out-of-range fields
    and resets to the defaults (all zero: the library's own choice, a 2 s wait
    bound) with NULL.  Host-only calls."""
    try:
        pk.kamera_set_launch_tuning(bn=128, stages=3, uv_slots=1, ksplit=2, no_pdl=1, grid=40,
                                    wait_limit_ns=1_000_000, test_unarm_first_stage=1)
        t = pk.kamera_get_launch_tuning()
        assert (t.bn, t.stages, t.uv_slots, t.ksplit, t.no_pdl, t.grid, t.wait_limit_ns,
                t.test_unarm_first_stage) == (128, 3, 1, 2, 1, 40, 1_000_000, 1)
        for bad in ({"bn": 96}, {"stages": 1}, {"stages": 7}, {"uv_slots": 9}, {"ksplit": 3}, {"grid": -1},
                    {"grid": 70000}, {"wait_limit_ns": 10}, {"wait_limit_ns": 61_000_000_000}, {"reserved": 1}):
            assert pk.kamera_set_launch_tuning(raise_on_error=False, **bad) == pk.KAMERA_ERR_INVALID_ARG, bad
        # a rejected setting leaves the previous one in place
        assert pk.kamera_get_launch_tuning().bn == 128
        assert lib.kamera_get_launch_tuning(None) == pk.KAMERA_ERR_NULL
    finally:
        pk.kamera_set_launch_tuning()
    t = pk.kamera_get_launch_tuning()
    assert all(getattr(t, f) == 0 for f, _ in t._fields_)


def test_orbit_mean_validation(lib):
    assert pk.kamera_orbit_mean(FAKE, 0, 100, 100, FAKE + (1 << 20), None, False) == pk.KAMERA_ERR_INVALID_ARG
    assert pk.kamera_orbit_mean(FAKE, 3, 50, 100, FAKE + (1 << 20), None, False) == pk.KAMERA_ERR_INVALID_ARG
    assert pk.kamera_orbit_mean(None, 3, 100, 100, FAKE + (1 << 20), None, False) == pk.KAMERA_ERR_NULL
    assert pk.kamera_orbit_mean(FAKE, 3, 100, 100, FAKE + 4, None, False) == pk.KAMERA_ERR_INVALID_ARG  # overlap
    assert pk.kamera_orbit_mean(FAKE + 2, 3, 100, 100, FAKE + (1 << 20), None, False) == pk.KAMERA_ERR_ALIGNMENT
    assert pk.kamera_orbit_mean(FAKE, 3, 100, 0, FAKE, None, False) == pk.KAMERA_OK


# ---- compressed canonical store ---------------------------------------------------------------------

def test_v_codebook_matches_the_oracle_bit_for_bit(lib):
    """The library's Lloyd-Max solver and the oracle's are written separately;
    the fp32 codebook and thresholds (part of the store format) must agree."""
    import numpy as np

    import oracle

    c_lib, t_lib = pk.kamera_v_codebook()
    c_or, t_or = oracle.v_codebook()
    np.testing.assert_array_equal(c_lib.view(np.uint32), c_or.view(np.uint32))
    np.testing.assert_array_equal(t_lib.view(np.uint32), t_or.view(np.uint32))


def _cstore(**kw):
    c = pk.kamera_compressed_store(FAKE, FAKE + 1024, FAKE + 4096, FAKE + 8192, FAKE + 16384, FAKE + 20480, 4, 0,
                                   1 << 16)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _reuse_c(model, pool, cs=None, n=1):
    return pk.kamera_reuse_compressed(model, cs if cs is not None else _cstore(), None, FAKE, n, pool, None, None,
                                      raise_on_error=False)


def test_compressed_validation(lib):
    assert pk.kamera_reuse_compressed(_gqa_model(), None, None, FAKE, 1, _pool(), None, None,
                                      False) == pk.KAMERA_ERR_NULL
    assert _reuse_c(_gqa_model(), _pool(), _cstore(v_norm=None)) == pk.KAMERA_ERR_NULL
    assert _reuse_c(_gqa_model(), _pool(), _cstore(k_codes=FAKE + 8)) == pk.KAMERA_ERR_ALIGNMENT
    assert _reuse_c(_gqa_model(), _pool(), _cstore(row_offset=FAKE + 4)) == pk.KAMERA_ERR_ALIGNMENT
    assert _reuse_c(_gqa_model(), _pool(), _cstore(reserved=1)) == pk.KAMERA_ERR_INVALID_ARG
    assert _reuse_c(_gqa_model(), _pool(), _cstore(n_rows=1 << 31)) == pk.KAMERA_ERR_UNSUPPORTED
    mla = pk.model_desc(pk.KAMERA_MLA, 2, rope_dim=64, latent_dim=512)
    assert _reuse_c(mla, _pool(v=None)) == pk.KAMERA_ERR_UNSUPPORTED
    assert _reuse_c(_gqa_model(head_dim=256), _pool()) == pk.KAMERA_ERR_UNSUPPORTED
    assert _reuse_c(_gqa_model(head_dim=64, num_kv_heads=1), _pool()) == pk.KAMERA_ERR_UNSUPPORTED  # D = 64
    assert _reuse_c(_gqa_model(), _pool(), n=0) == pk.KAMERA_OK


def test_compress_chunks_validation(lib):
    def run(model, src, dst):
        return pk.kamera_compress_chunks(model, src, dst, None, None, raise_on_error=False)

    assert run(None, _store(), _cstore()) == pk.KAMERA_ERR_NULL
    mla = pk.model_desc(pk.KAMERA_MLA, 2, rope_dim=64, latent_dim=512)
    assert run(mla, _store(), _cstore()) == pk.KAMERA_ERR_UNSUPPORTED
    assert run(_gqa_model(head_dim=192), _store(), _cstore()) == pk.KAMERA_ERR_UNSUPPORTED
    assert run(_gqa_model(), _store(), _cstore(n_chunks=3)) == pk.KAMERA_ERR_INVALID_ARG
    assert run(_gqa_model(), _store(), _cstore(v_codes=None)) == pk.KAMERA_ERR_NULL
    assert run(_gqa_model(), _store(), _cstore(v_codes=FAKE + 8)) == pk.KAMERA_ERR_ALIGNMENT
    empty = pk.kamera_chunk_store(None, 0, None, None, 0)
    assert run(_gqa_model(), empty, _cstore(n_chunks=0)) == pk.KAMERA_OK


def test_binding_fails_loudly_without_the_library(tmp_path):
    """With no built library there is no other path: loading and every call
    raise ImportError (checked in a fresh interpreter so that this process's
    loaded library is not disturbed)."""
    code = (
        "import sys\n"
        f"sys.path.insert(0, {os.path.dirname(_build.PKG)!r})\n"
        "import position_invariant_kv_kamera_gb300 as pk\n"
        "from position_invariant_kv_kamera_gb300 import _build\n"
        f"_build.LIB = {str(tmp_path / 'libkamera.so')!r}\n"
        "for f in (pk.load, pk.abi_version, pk.kamera_v_codebook):\n"
        "    try:\n"
        "        f()\n"
        "    except ImportError:\n"
        "        continue\n"
        "    sys.exit('no error from ' + f.__name__)\n"
    )
    r = subprocess.run([os.sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr


def test_callable_from_plain_c(lib, tmp_path):
    """A C program (gcc, no CUDA headers) links against the library and calls
    it through the header alone: version, codebook, and a validation error
    with its message (no GPU needed: the call returns before any CUDA call)."""
    prog = tmp_path / "client.c"
    prog.write_text(r'''
#include <stdio.h>
#include "kamera.h"
int main(void) {
  float c[8], t[7];
  if (kamera_abi_version() != KAMERA_ABI_VERSION) return 1;
  if (kamera_v_codebook(c, t) != KAMERA_OK) return 2;
  for (int k = 0; k < 4; ++k) if (c[7 - k] != -c[k] || !(c[k] < c[k + 1])) return 3;
  kamera_status s = kamera_reuse_batched(NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL);
  printf("%s|%s|%.4f\n", kamera_status_string(s), kamera_last_error(), c[7]);
  return s == KAMERA_ERR_NULL ? 0 : 4;
}
''')
    exe = tmp_path / "client"
    libdir = os.path.dirname(_build.LIB)
    subprocess.run(["gcc", "-std=c11", "-I" + _build.INCLUDE, "-o", str(exe), str(prog), "-L" + libdir, "-lkamera",
                    "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    status, msg, c7 = r.stdout.strip().split("|")
    assert status == "KAMERA_ERR_NULL" and "NULL" in msg and abs(float(c7) - 2.152) < 1e-3


def test_every_cuda_build_targets_sm_103a_only():
    """The library's units, its link and the generator's device twin are
    built for sm_103a alone (one -gencode, no PTX for other targets)."""
    from synth import device as synth_device

    cmds = [_build.compile_cmd(s) for s in _build.SOURCES] + [_build.link_cmd(), synth_device.build_cmd()]
    for cmd in cmds:
        gencodes = [cmd[i + 1] for i, a in enumerate(cmd) if a == "-gencode"]
        assert gencodes == ["arch=compute_103a,code=sm_103a"], cmd
        assert not any(a.startswith(("-arch", "--gpu-architecture", "-code")) for a in cmd), cmd
    for cmd in cmds[:-2]:
        assert "-lineinfo" in cmd and "-O3" in cmd
