"""CPU-only checks of the C-ABI library: it builds, loads, exports every
declared entry point, its ctypes structs match the C layout, and host-side
argument checks reject bad calls before anything is launched."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    import glob
    from sparse_attention_prolog_gb300 import binding, build
    srcs = glob.glob(os.path.join(build.CSRC, "*")) + [HEADER]
    if not os.path.exists(binding.LIB_PATH) or \
            os.path.getmtime(binding.LIB_PATH) < max(os.path.getmtime(s) for s in srcs):
        build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dsa.h but not exported"
    from sparse_attention_prolog_gb300 import binding
    assert set(binding.EXPORTS) <= set(names)


def test_struct_layout_matches_header(lib, tmp_path):
    from sparse_attention_prolog_gb300 import binding as B
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "dsa.h"', "int main(void) {"]
    for cname, py in (("dsa_prolog_args", B.PrologArgs), ("dsa_topk_args", B.TopkArgs),
                      ("dsa_attn_args", B.AttnArgs), ("dsa_act_quant_args", B.ActQuantArgs),
                      ("dsa_int8_gemm_args", B.Int8GemmArgs), ("dsa_mhc_args", B.MhcArgs),
                      ("dsa_mla_prolog_args", B.MlaArgs)):
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0; }")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(line.split() for line in out if line)
    for cname, py in (("dsa_prolog_args", B.PrologArgs), ("dsa_topk_args", B.TopkArgs),
                      ("dsa_attn_args", B.AttnArgs), ("dsa_act_quant_args", B.ActQuantArgs),
                      ("dsa_int8_gemm_args", B.Int8GemmArgs), ("dsa_mhc_args", B.MhcArgs),
                      ("dsa_mla_prolog_args", B.MlaArgs)):
        assert int(got[cname]) == ctypes.sizeof(py)
        for f, _ in py._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(py, f).offset, f"{cname}.{f}"


def test_status_strings(lib):
    from sparse_attention_prolog_gb300 import binding as B
    assert B.status_string(0) == "ok"
    assert "workspace" in B.status_string(3)
    assert lib.dsa_abi_version() == 104
    assert "timed out" in B.status_string(5)
    assert "device-side data" in B.status_string(6)
    assert B.status_string(7) == "unknown status"


def test_host_validation_rejects_before_launch(lib):
    from sparse_attention_prolog_gb300 import binding as B
    null = ctypes.c_void_p(0)
    assert lib.dsa_indexer_prolog(None, null, 0, null) == 1
    a = B.PrologArgs()
    a.T, a.H_I, a.d_I, a.d_rope, a.K_q, a.D_x, a.rope_max_pos = 8, 64, 96, 64, 1536, 7168, 10
    assert lib.dsa_indexer_prolog(ctypes.byref(a), null, 0, null) == 2      # d_I 96 unsupported
    a.d_I = 128
    a.T = 33
    assert lib.dsa_indexer_prolog(ctypes.byref(a), null, 0, null) == 2      # too many tokens
    a.T = 8
    assert lib.dsa_indexer_prolog(ctypes.byref(a), null, 0, null) == 1      # null tensors
    a.T = 0
    assert lib.dsa_indexer_prolog(ctypes.byref(a), null, 0, null) == 0      # empty: no-op
    t = B.TopkArgs()
    t.T, t.B, t.n_q, t.H_I, t.d_I, t.topk, t.max_L = 8, 4, 3, 64, 128, 2048, 65536
    assert lib.dsa_indexer_topk(ctypes.byref(t), null, 0, null) == 1        # T != B * n_q
    t.n_q = 2
    t.max_L = 1000
    assert lib.dsa_indexer_topk(ctypes.byref(t), null, 0, null) == 2        # max_L % 128
    t.max_L, t.H_I = 65536, 48
    assert lib.dsa_indexer_topk(ctypes.byref(t), null, 0, null) == 2        # H_I 48
    t.H_I = 64
    assert lib.dsa_indexer_topk(ctypes.byref(t), null, 0, null) == 1        # null tensors
    assert lib.dsa_indexer_topk_workspace(ctypes.byref(t)) == 0            # invalid -> 0
    base = 1 << 20  # fake, suitably aligned device addresses: only validated, never read
    for i, f in enumerate(("q", "q_scale", "w", "k_cache", "k_scale", "pos", "topk_idx")):
        setattr(t, f, base + i * 4096)
    assert lib.dsa_indexer_topk_workspace(ctypes.byref(t)) > 0             # valid -> scores + histograms
    t.k_scale = base + 4 * 4096 + 2
    assert lib.dsa_indexer_topk_workspace(ctypes.byref(t)) == 0            # k_scale must be 16-byte aligned
    assert lib.dsa_indexer_topk(ctypes.byref(t), null, 0, null) == 1
    # a per-token sequence map lifts T == B * n_q (n_q is then ignored)
    t.k_scale = base + 4 * 4096
    t.T, t.n_q = 7, 3
    assert lib.dsa_indexer_topk_workspace(ctypes.byref(t)) == 0            # no map: 7 != 4 * 3
    t.seq_of_token = base + 9 * 4096
    assert lib.dsa_indexer_topk_workspace(ctypes.byref(t)) > 0             # with a map: valid
    t.seq_of_token = base + 9 * 4096 + 2
    assert lib.dsa_indexer_topk_workspace(ctypes.byref(t)) == 0            # map not 4-byte aligned
    t.seq_of_token, t.T = base + 9 * 4096, 65536
    assert lib.dsa_indexer_topk(ctypes.byref(t), null, 0, null) == 2        # a map covers < 65536 tokens
    at = B.AttnArgs()
    at.T, at.B, at.n_q, at.H, at.d_qk, at.d_v, at.topk, at.max_L, at.scale = 8, 4, 2, 128, 512, 512, 2048, 65536, 0.07
    assert lib.dsa_sparse_attn(ctypes.byref(at), null, 0, null) == 2        # d_qk 512
    at.d_qk = 576
    assert lib.dsa_sparse_attn(ctypes.byref(at), null, 0, null) == 1        # null tensors
    at.T = 0
    assert lib.dsa_sparse_attn(ctypes.byref(at), null, 0, null) == 0
    for i, f in enumerate(("q", "kv", "topk_idx", "out")):
        setattr(at, f, base + i * 4096)
    at.T, at.n_q = 7, 5
    assert lib.dsa_sparse_attn_workspace(ctypes.byref(at)) == 0             # no map: 7 != 4 * 5
    at.seq_of_token = base + 9 * 4096
    # past the argument checks: what follows needs a GPU (workspace or CUDA status here)
    assert lib.dsa_sparse_attn(ctypes.byref(at), null, 0, null) in (0, 3, 4)
    at.seq_of_token = 0
    assert lib.dsa_indexer_prolog_noalloc(None, null) == 1                 # the no-allocation entry: null args
    assert lib.dsa_act_quant(None, null) == 1
    aq = B.ActQuantArgs(4, 100, 1 << 20, 1 << 21, 1 << 22, 0)
    assert lib.dsa_act_quant(ctypes.byref(aq), null) == 2                  # N % 8
    aq.N = 64
    aq.x = (1 << 20) + 8
    assert lib.dsa_act_quant(ctypes.byref(aq), null) == 1                  # x not 16-byte aligned
    aq.M = 0
    assert lib.dsa_act_quant(ctypes.byref(aq), null) == 0                  # empty: no-op
    g = B.Int8GemmArgs(8388609, 64, 128, 1 << 20, 1 << 21, 1 << 22, 1 << 23, 1 << 24)
    assert lib.dsa_int8_gemm(ctypes.byref(g), null) == 2                   # M > 2^23
    g.M, g.K = 8, 100
    assert lib.dsa_int8_gemm(ctypes.byref(g), null) == 2                   # K % 16
    g.K, g.b = 128, (1 << 22) + 4
    assert lib.dsa_int8_gemm(ctypes.byref(g), null) == 1                   # b not 16-byte aligned
    g.N = 0
    assert lib.dsa_int8_gemm(ctypes.byref(g), null) == 0                   # empty: no-op
    h = B.MhcArgs(16, 6, 5, 1e-6, 1 << 20, 1 << 21, 1 << 22, 1 << 23, 1 << 24, 1 << 25)
    assert lib.dsa_mhc(ctypes.byref(h), null) == 2                         # hc 6
    h.hc, h.eps = 4, -1.0
    assert lib.dsa_mhc(ctypes.byref(h), null) == 1                         # negative eps
    h.eps, h.comb = 1e-6, (1 << 25) + 4
    assert lib.dsa_mhc(ctypes.byref(h), null) == 1                         # comb not 16-byte aligned
    h.eps, h.n = 1e-6, 0
    assert lib.dsa_mhc(ctypes.byref(h), null) == 0                         # empty: no-op
    ptrs = [(1 << 20) * (i + 1) for i in range(16)]
    m = B.MlaArgs(8, 128, 1536, 7168, 1e-6, 4096, 0, *ptrs, 64)
    ws = ctypes.c_void_p(1 << 30)
    need = lib.dsa_mla_prolog_workspace(ctypes.byref(m))
    assert need >= 8 * (1536 + 576) * 4 + 8 * 128 * 128 * 4
    assert lib.dsa_mla_prolog(ctypes.byref(m), null, 0, null) == 3          # no workspace
    m.T = 33
    assert lib.dsa_mla_prolog(ctypes.byref(m), ws, need, null) == 2         # T > 32
    m.T, m.K_q = 8, 1000
    assert lib.dsa_mla_prolog(ctypes.byref(m), ws, need, null) == 2         # K_q % 128
    m.K_q, m.H = 1536, 0
    assert lib.dsa_mla_prolog(ctypes.byref(m), ws, need, null) == 1         # no heads
    m.H, m.q = 128, (1 << 20) * 18 + 4
    assert lib.dsa_mla_prolog(ctypes.byref(m), ws, need, null) == 1         # q not 16-byte aligned
    m.T = 0
    assert lib.dsa_mla_prolog(ctypes.byref(m), null, 0, null) == 0          # empty: no-op
    assert lib.dsa_set_wait_limit_ns(61 * 10 ** 9) == 1                     # wait limit beyond 60 s


def test_missing_library_fails_loudly(tmp_path):
    from sparse_attention_prolog_gb300 import binding as B
    with pytest.raises(B.DSAError):
        _fresh_load(B, str(tmp_path / "nope.so"))


def _fresh_load(B, path):
    saved = B._lib
    B._lib = None
    try:
        B.load(path)
    finally:
        B._lib = saved


def test_plain_c_program_links_and_calls_the_abi(lib, tmp_path):
    """The boundary is a C ABI: a C program compiled against dsa.h and
    linked to libdsa.so reads the version and status strings and gets the
    host-side rejections (nothing is launched on these paths)."""
    from sparse_attention_prolog_gb300 import binding
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "dsa.h"
int main(void) {
  if (dsa_abi_version() < 100) return 10;
  if (strcmp(dsa_status_string(DSA_OK), "ok") != 0) return 11;
  if (strcmp(dsa_status_string(42), "unknown status") != 0) return 12;
  dsa_mhc_args m;
  memset(&m, 0, sizeof m);
  m.n = 4; m.hc = 6; m.iters = 1; m.eps = 1e-6f;
  if (dsa_mhc(&m, NULL) != DSA_ERR_UNSUPPORTED) return 13;           /* hc 6 */
  dsa_mla_prolog_args a;
  memset(&a, 0, sizeof a);
  a.T = 8; a.H = 128; a.K_q = 1536; a.D_x = 7168; a.rope_max_pos = 1;
  if (dsa_mla_prolog(&a, NULL, 0, NULL) != DSA_ERR_INVALID_ARG) return 14;  /* null pointers */
  if (dsa_mla_prolog_workspace(&a) != 0) return 15;                  /* invalid: no size */
  a.T = 0;
  if (dsa_mla_prolog(&a, NULL, 0, NULL) != DSA_OK) return 16;        /* empty: no-op */
  dsa_act_quant_args q;
  memset(&q, 0, sizeof q);
  q.M = 2; q.N = 7;
  if (dsa_act_quant(&q, NULL) != DSA_ERR_UNSUPPORTED) return 17;     /* N % 8 */
  printf("ok\n");
  return 0;
}
""")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(binding.LIB_PATH)
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", libdir, "-ldsa",
                    f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
