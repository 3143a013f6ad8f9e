"""Host-side tests of libspfuse that need no GPU: the library builds for
sm_103a, loads, exports every entry point include/spfuse.h declares, and
rejects invalid arguments before touching the device."""
import ctypes
import os
import re
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spfuse.h")


@pytest.fixture(scope="module")
def spf():
    from residual_sp_rs_gb300 import build, ops
    build.build()
    return ops


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(sp\w*|hp2sp)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["sp_rs_dropout_residual_norm_fwd", "sp_rs_dropout_residual_norm_fwd_rows",
              "sp_rs_dropout_residual_norm_bwd_rows",
              "sp_rs_bwd_workspace_bytes",
              "sp_rs_dropout_residual_norm_bwd", "sp2hp", "hp2sp", "sp_status_string", "sp_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(spf):
    lib = spf.lib()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", spf.LIB_PATH], capture_output=True, text=True)
    if out.returncode == 0:
        exported = {l.split()[-1] for l in out.stdout.splitlines() if l.strip()}
        for n in declared_functions():
            assert n in exported, n


def test_library_is_built_for_sm_103a_only():
    from residual_sp_rs_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_library_matches_the_sources(spf):
    """The library reports the hash of the sources it was built from, and the
    binding refuses one whose hash is not the tree's."""
    from residual_sp_rs_gb300 import build
    L = spf.lib()
    assert L.sp_build_hash().decode() == build.source_hash()
    with pytest.raises(RuntimeError, match="stale"):
        spf._verify_hash(L, "0" * 64)


def test_struct_layout_matches_header(spf):
    assert ctypes.sizeof(spf.SpRsDesc) == 72
    assert spf.SpRsDesc.seed.offset == 48 and spf.SpRsDesc.nshards.offset == 56
    assert spf.SpRsDesc.status.offset == 64
    assert ctypes.sizeof(spf.SpKernelPlan) == 80 and spf.SpKernelPlan.workspace_bytes.offset == 72


def test_status_strings(spf):
    for code in range(8):
        assert spf.status_string(code).startswith("SP_")
    assert spf.lib().sp_version() >= 100


FAKE = 1 << 20   # a 16-byte aligned address that is never dereferenced


def _fwd(spf, desc, partials=None, residual=FAKE, gamma=FAKE, beta=FAKE, h=FAKE, y=FAKE, mask=FAKE,
         rstd=FAKE, mean=FAKE):
    partials = [FAKE] * desc.T if partials is None else partials
    arr = (ctypes.c_void_p * max(1, len(partials)))(*partials)
    return spf.lib().sp_rs_dropout_residual_norm_fwd(ctypes.byref(desc), arr, residual, gamma, beta,
                                                    h, y, mask, rstd, mean, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), 1), (dict(T=9), 1), (dict(j=2), 1), (dict(j=-1), 1), (dict(nshards=3), 1),
    (dict(p=1.0), 1), (dict(p=-0.1), 1), (dict(p=float("nan")), 1), (dict(eps=0.0), 1),
    (dict(eps=float("inf")), 1), (dict(S=15), 2), (dict(H=12), 2), (dict(H=16392), 2),
    (dict(S=-2), 2), (dict(dtype=7), 4), (dict(norm=3), 4),
])
def test_fwd_rejects_bad_descriptors(spf, kw, code):
    base = dict(T=2, j=0, S=16, B=2, H=64, dtype="bf16", norm="rms", p=0.1, eps=1e-6, seed=0)
    base.update(kw)
    desc = spf.make_desc(**base)
    assert _fwd(spf, desc) == code


def test_fwd_rejects_bad_pointers(spf):
    d = spf.make_desc(2, 0, 16, 2, 64, "bf16", "ln", 0.1, 1e-5)
    assert _fwd(spf, d, partials=[FAKE, 0]) == 1
    assert _fwd(spf, d, residual=0) == 1
    assert _fwd(spf, d, beta=0) == 1            # LayerNorm needs beta
    assert _fwd(spf, d, mean=0) == 1            # ... and mean
    assert _fwd(spf, d, mask=0) in (0, 6)       # no stored mask: accepted (6 = no GPU here)
    assert _fwd(spf, d, partials=[FAKE, FAKE + 8]) == 3
    assert _fwd(spf, d, y=FAKE + 2) == 3
    assert _fwd(spf, d, rstd=FAKE + 2) == 3
    d0 = spf.make_desc(2, 0, 16, 2, 64, "bf16", "rms", 0.0, 1e-5)
    d0.reserved = 1
    assert _fwd(spf, d0) == 1
    d1 = spf.make_desc(2, 0, 16, 2, 64, "bf16", "rms", 0.0, 1e-5)
    d1.status = FAKE + 2                        # the status word must be 4-byte aligned
    assert _fwd(spf, d1) == 3


def _fwd_rows(spf, desc, row_begin, row_count, partials=None, mask=FAKE, ptr=FAKE):
    partials = [ptr] * desc.T if partials is None else partials
    arr = (ctypes.c_void_p * max(1, len(partials)))(*partials)
    return spf.lib().sp_rs_dropout_residual_norm_fwd_rows(
        ctypes.byref(desc), row_begin, row_count, arr, ptr, ptr, ptr, ptr, ptr, mask, ptr, ptr, None)


def test_fwd_rows_validates_the_range(spf):
    # T=2, S=16, B=2: 16 rows in the call; H=24 bf16 (48-byte rows, 24-byte mask rows)
    d = spf.make_desc(2, 0, 16, 2, 24, "bf16", "rms", 0.1, 1e-6)
    for rb, rc in [(-1, 4), (0, -1), (17, 0), (10, 7), (1 << 62, 1 << 62)]:
        assert _fwd_rows(spf, d, rb, rc) == 1, (rb, rc)
    assert _fwd_rows(spf, d, 16, 0) == 0          # an empty range at the end
    assert _fwd_rows(spf, d, 3, 0, ptr=0) == 0    # empty: no pointer is checked or touched
    assert _fwd_rows(spf, d, 0, 4, ptr=0) == 1    # a real range needs its pointers
    # the range's first mask row must stay 16-byte aligned: row 1 starts 24 bytes in
    assert _fwd_rows(spf, d, 1, 4) == 3
    assert _fwd_rows(spf, d, 1, 4, mask=0) in (0, 6)   # no stored mask: accepted (6 = no GPU)
    assert _fwd_rows(spf, d, 2, 4) in (0, 6)           # row 2 starts 48 bytes in
    # nshards = T: the range runs over both shards' rows
    d2 = spf.make_desc(2, 0, 16, 2, 24, "bf16", "rms", 0.1, 1e-6, 0, 2)
    assert _fwd_rows(spf, d2, 30, 3) == 1
    assert _fwd_rows(spf, d2, 30, 2) in (0, 6)


def test_empty_problem_launches_nothing(spf):
    d = spf.make_desc(2, 0, 0, 2, 64, "bf16", "rms", 0.1, 1e-6)
    assert _fwd(spf, d) == 0   # S = 0: nothing to do, no device touched


def test_bwd_rejects_bad_arguments(spf):
    L = spf.lib()
    d = spf.make_desc(2, 0, 16, 2, 64, "bf16", "rms", 0.1, 1e-6)

    def call(desc, mask=FAKE, dy=FAKE, ws=FAKE, nbytes=1 << 30):
        return L.sp_rs_dropout_residual_norm_bwd(ctypes.byref(desc), dy, FAKE, FAKE, FAKE, mask, FAKE,
                                                 FAKE, FAKE, FAKE, FAKE, FAKE, ws, nbytes, None)
    assert call(d, mask=0) in (0, 6)            # regenerated mask: accepted (6 = no GPU here)
    assert call(d, dy=0) == 1
    assert call(d, dy=FAKE + 4) == 3
    bad = spf.make_desc(3, 0, 16, 2, 64, "bf16", "rms", 0.1, 1e-6)
    assert call(bad) == 2
    assert L.sp_rs_bwd_workspace_bytes(ctypes.byref(bad)) == 0


def test_bwd_rows_validates_the_range(spf):
    L = spf.lib()
    # T=2, S=16, B=2: 16 rows in the call; H=24 bf16 (48-byte rows, 24-byte mask rows)
    d = spf.make_desc(2, 0, 16, 2, 24, "bf16", "rms", 0.1, 1e-6)

    def call(rb, rc, acc=0, mask=FAKE, ptr=FAKE):
        return L.sp_rs_dropout_residual_norm_bwd_rows(ctypes.byref(d), rb, rc, acc, ptr, ptr, ptr, ptr, mask,
                                                      ptr, ptr, ptr, ptr, FAKE, FAKE, FAKE, 1 << 30, None)
    for rb, rc in [(-1, 4), (0, -1), (17, 0), (10, 7), (1 << 62, 1 << 62)]:
        assert call(rb, rc) == 1, (rb, rc)
    assert call(16, 0, acc=1) == 0              # empty and accumulating: nothing launched
    assert call(3, 0, acc=1, ptr=0) == 0        # ... and no per-row pointer needed
    assert call(0, 4, ptr=0) == 1
    assert call(1, 4) == 3                      # row 1's mask bytes start 24 bytes in
    assert call(1, 4, mask=0) in (0, 6)         # regenerated mask: accepted (6 = no GPU)
    assert call(2, 4) in (0, 6)


@pytest.mark.parametrize("args,code", [
    ((FAKE, FAKE, 16, 64, 4, 9), 4), ((0, FAKE, 16, 64, 4, 1), 1), ((FAKE, FAKE, 15, 64, 4, 1), 2),
    ((FAKE, FAKE, 16, 48, 4, 1), 2), ((FAKE, FAKE, 16, 64, 9, 1), 1), ((FAKE + 4, FAKE, 16, 64, 4, 1), 3),
])
def test_layout_rejects_bad_arguments(spf, args, code):
    L = spf.lib()
    assert L.sp2hp(*args, None) == code
    assert L.hp2sp(*args, None) == code


def test_launch_failure_is_reported(spf):
    """A failing launch (injected on the host) comes back as SP_ERR_CUDA."""
    code = textwrap.dedent(f"""
        import ctypes, sys
        sys.path.insert(0, {ROOT!r})
        from residual_sp_rs_gb300 import ops
        d = ops.make_desc(2, 0, 16, 2, 64, "bf16", "rms", 0.1, 1e-6)
        arr = (ctypes.c_void_p * 2)({FAKE}, {FAKE})
        L = ops.lib()
        r1 = L.sp_rs_dropout_residual_norm_fwd(ctypes.byref(d), arr, {FAKE}, {FAKE}, None, {FAKE},
                                               {FAKE}, {FAKE}, {FAKE}, None, None)
        r2 = L.sp2hp({FAKE}, {FAKE}, 16, 64, 4, 1, None)
        print(r1, r2)
    """)
    env = dict(os.environ, SPFUSE_FAIL_LAUNCH="1")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["6", "6"]


def test_python_binding_raises_on_error(spf):
    d = spf.make_desc(2, 0, 15, 2, 64, "bf16", "rms", 0.1, 1e-6)
    with pytest.raises(RuntimeError, match="SP_ERR_SHAPE"):
        spf.sp_rs_dropout_residual_norm_fwd(d, [FAKE, FAKE], FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE,
                                            None, stream=0)


def test_product_package_does_not_import_oracle():
    """The product path never reaches the oracle."""
    pkg = os.path.join(ROOT, "residual_sp_rs_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "oracle.h" not in txt and "liboracle" not in txt, f


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "spfuse.h"

int main(void) {
  sp_rs_desc_t d;
  sp_plan_info_t info;
  memset(&d, 0, sizeof d);
  d.T = 2; d.j = 0; d.S = 2048; d.B = 2; d.H = 768;
  d.dtype = SP_BF16; d.norm = SP_RMSNORM; d.p = 0.1f; d.eps = 1e-6f; d.seed = 0; d.nshards = 2;
  if (sp_plan_describe(&d, 152, 232448, 1, 1, &info) != SP_OK) return 1;
  printf("version %d fwd_block %d bwd_block %d bwd_ws %lld\n", (int)sp_version(), (int)info.fwd.block,
         (int)info.bwd.block, (long long)info.bwd.workspace_bytes);
  d.T = 0;  /* invalid: refused before anything touches a device */
  printf("invalid %d %s\n", (int)sp_rs_dropout_residual_norm_fwd(&d, NULL, NULL, NULL, NULL, NULL, NULL,
                                                                  NULL, NULL, NULL, NULL),
         sp_status_string(SP_ERR_INVALID_ARG));
  printf("workspace %lu\n", (unsigned long)sp_rs_bwd_workspace_bytes(&d));
  return 0;
}
"""


def test_header_is_plain_c_and_links(spf, tmp_path):
    """The boundary is a C ABI: a C11 program compiled with warnings as errors
    includes the header, links libspfuse and calls entry points that need no
    GPU (launch plans, validation, status strings)."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(spf.LIB_PATH)
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{os.path.join(ROOT, 'include')}",
                        str(src), "-o", str(exe), f"-L{libdir}", "-l:" + os.path.basename(spf.LIB_PATH),
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.split("\n")
    assert lines[0].startswith("version ") and "fwd_block 896" in lines[0] and "bwd_block 512" in lines[0]
    assert lines[1].startswith("invalid 1 SP_ERR_INVALID_ARG")
    assert lines[2] == "workspace 0"
