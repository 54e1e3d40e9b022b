"""The C-ABI library: it loads without a GPU, exports every entry point the
header declares (and nothing internal), and rejects invalid arguments with
the documented status codes before touching the device. CPU only."""
import ctypes
import os
import re
import subprocess

import pytest

import moe_expert_layer_grouped_gb300 as moe
from moe_expert_layer_grouped_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return moe.load()


def test_every_source_and_header_is_a_build_input():
    # a file left out would either not be compiled or, for a header, not
    # trigger a rebuild when only it changed
    files = os.listdir(cuda_build.SRC)
    assert sorted(f for f in files if f.endswith(".cu")) == sorted(cuda_build.SOURCES)
    assert sorted(f for f in files if f.endswith((".cuh", ".h"))) == sorted(cuda_build.HEADERS)


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """The header is plain C (C11, pedantic, warnings as errors) and a C program
    links against the library and calls it: no device work, the gate call is
    rejected by host validation."""
    src = tmp_path / "use_abi.c"
    src.write_text(r"""
#include <stdio.h>
#include "moe_gb300.h"
int main(void) {
  int v = moe_abi_version();
  const char* s = moe_status_string(MOE_ERR_WORKSPACE);
  /* E % num_groups != 0 */
  moe_status st = moe_gate((const float*)0x10000, NULL, 4, 10, 3, 1, 2, MOE_SCORE_SIGMOID, 1,
                           1.0f, (int32_t*)0x10000, (float*)0x10000, NULL);
  printf("%d %s %d\n", v, s, (int)st);
  return st == MOE_ERR_INVALID_ARG ? 0 : 1;
}
""")
    so = cuda_build.build()
    exe = tmp_path / "use_abi"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.dirname(HEADER), str(src), so,
                    "-Wl,-rpath," + os.path.dirname(so), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    version, name, status = r.stdout.split()
    assert int(version) == lib.moe_abi_version() and name == "MOE_ERR_WORKSPACE"
    assert int(status) == INVALID


def test_product_and_oracle_share_no_code():
    """The CUDA library and its binding never import, include or load the
    oracle, and the oracle never touches the library's package or sources
    (the seeded input generator, synth.py, is the one module both sides use,
    and it does not import the oracle either)."""
    pkg = os.path.join(ROOT, "moe_expert_layer_grouped_gb300")
    to_oracle = re.compile(r"^\s*(import oracle|from oracle)|liboracle|oracle\.h|oracle_build",
                           re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not to_oracle.search(text), os.path.join(dirpath, f)
    to_product = re.compile(r"moe_expert_layer_grouped_gb300|moe_gb300\.h|csrc|libmoe_gb300")
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        if f.endswith((".py", ".c", ".h")):
            assert not to_product.search(open(os.path.join(odir, f)).read()), f


def _oracle_imports(path):
    """(enclosing function or None, line) of every import of the oracle package."""
    import ast
    tree = ast.parse(open(path).read())
    found = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            mods = []
            if isinstance(child, ast.Import):
                mods = [a.name for a in child.names]
            elif isinstance(child, ast.ImportFrom):
                mods = [child.module or ""]
            if any(m == "oracle" or m.startswith("oracle.") for m in mods):
                found.append((name, child.lineno))
            visit(child, name)

    visit(tree, None)
    return found


def test_only_test_smoke_and_baseline_code_use_the_oracle():
    # outside tests/: smoke() checks against it, build() compiles it, and
    # the benchmark times it in its CPU-baseline and reference legs
    allowed = {"__graft_entry__.py": {"smoke", "build"},
               "bench.py": {"cpu_baseline", "run_reference"}}
    for dirpath, dirs, files in os.walk(ROOT):
        rel = os.path.relpath(dirpath, ROOT)
        dirs[:] = [d for d in dirs if not d.startswith((".", "_")) and d not in ("tests", "oracle")]
        for f in files:
            if not f.endswith(".py"):
                continue
            key = f if rel == "." else os.path.join(rel, f)
            for fn, line in _oracle_imports(os.path.join(dirpath, f)):
                assert fn in allowed.get(key, set()), f"{key}:{line} imports the oracle in {fn}"


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["moe_gate", "moe_permute_quant", "moe_grouped_gemm", "moe_act_quant",
                 "moe_unpermute_sum", "moe_forward", "moe_forward_host", "moe_workspace_size",
                 "moe_permute_workspace_size", "moe_device_status", "moe_status_string",
                 "moe_abi_version", "moe_forward_shared", "moe_forward_shared_host",
                 "moe_permute_quant_block", "moe_grouped_gemm_block", "moe_act_quant_block",
                 "moe_block_workspace_size", "moe_forward_block", "moe_forward_block_host",
                 "moe_test_gemm_timeout"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", moe.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(declared_functions()) <= exported
    # internal launchers stay hidden
    assert not any("launch_" in s for s in exported)


def test_status_strings_and_version(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(-3) == b"MOE_ERR_WORKSPACE"
    assert lib.moe_abi_version() >> 16 == 1


P = ctypes.c_void_p
GOOD = P(0x10000)      # aligned placeholders: never dereferenced, the calls
ODD = P(0x10008)       # below fail validation before any device work


def test_gate_argument_validation(lib):
    g = lib.moe_gate
    # E % G != 0, TG > G, K > TG*E/G, K > 32, E > 1024, bad scoring
    assert g(GOOD, None, 4, 10, 3, 1, 2, 0, 1, 1.0, GOOD, GOOD, None) == INVALID
    assert g(GOOD, None, 4, 8, 4, 5, 2, 0, 1, 1.0, GOOD, GOOD, None) == INVALID
    assert g(GOOD, None, 4, 8, 4, 1, 3, 0, 1, 1.0, GOOD, GOOD, None) == INVALID
    assert g(GOOD, None, 4, 64, 1, 1, 33, 0, 1, 1.0, GOOD, GOOD, None) == UNSUPPORTED
    assert g(GOOD, None, 4, 2048, 1, 1, 2, 0, 1, 1.0, GOOD, GOOD, None) == UNSUPPORTED
    assert g(GOOD, None, 4, 8, 1, 1, 2, 7, 1, 1.0, GOOD, GOOD, None) == INVALID
    # softmax takes no bias and no groups
    assert g(GOOD, GOOD, 4, 8, 1, 1, 2, 1, 1, 1.0, GOOD, GOOD, None) == UNSUPPORTED
    assert g(GOOD, None, 4, 8, 2, 1, 2, 1, 1, 1.0, GOOD, GOOD, None) == UNSUPPORTED
    # null / misaligned pointers
    assert g(None, None, 4, 8, 1, 1, 2, 0, 1, 1.0, GOOD, GOOD, None) == INVALID
    assert g(ODD, None, 4, 8, 1, 1, 2, 0, 1, 1.0, GOOD, GOOD, None) == INVALID
    assert g(GOOD, ODD, 4, 8, 1, 1, 2, 0, 1, 1.0, GOOD, GOOD, None) == INVALID


def test_permute_argument_validation(lib):
    f = lib.moe_permute_quant
    need = lib.moe_permute_workspace_size(100, 8, 2)
    assert need > 0
    args = lambda **kw: [kw.get("x", GOOD), GOOD, kw.get("T", 100), kw.get("H", 64), 8,
                         kw.get("K", 2), GOOD, GOOD, GOOD, GOOD, kw.get("ws", P(0x100000)),
                         kw.get("wsb", need), None]
    assert f(*args(H=48)) == INVALID                       # H % 32
    assert f(*args(K=33)) == UNSUPPORTED
    assert f(*args(H=32768)) == UNSUPPORTED
    assert f(*args(x=None)) == INVALID
    assert f(*args(wsb=need - 1)) == WORKSPACE
    assert f(*args(ws=None)) == WORKSPACE
    assert f(*args(ws=P(0x100010))) == WORKSPACE           # not 256-byte aligned


def test_gemm_act_unpermute_validation(lib):
    g = lib.moe_grouped_gemm
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 48, 64, 4, 0, GOOD, None, None) == INVALID
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 64, 48, 4, 0, GOOD, None, None) == INVALID
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 96, 64, 4, 1, GOOD, None, None) == INVALID
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 64, 64, 4, 2, GOOD, None, None) == INVALID
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 64, 64, 2048, 0, GOOD, None, None) == UNSUPPORTED
    assert g(ODD, GOOD, GOOD, GOOD, GOOD, 64, 64, 64, 4, 0, GOOD, None, None) == INVALID
    tg = lib.moe_test_gemm_timeout
    assert tg(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 64, 64, 4, 0, GOOD, -1, None) == INVALID
    assert tg(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 48, 64, 4, 0, GOOD, 2, None) == INVALID
    a = lib.moe_act_quant
    assert a(GOOD, None, 10, 48, GOOD, GOOD, None) == INVALID
    assert a(None, None, 10, 64, GOOD, GOOD, None) == INVALID
    u = lib.moe_unpermute_sum
    assert u(GOOD, GOOD, GOOD, 10, 2, 12, GOOD, None) == INVALID
    assert u(GOOD, GOOD, GOOD, 10, 40, 64, GOOD, None) == UNSUPPORTED


def test_forward_validation_and_workspace(lib):
    f = lib.moe_forward
    T, H, I, E, K = 16, 128, 64, 8, 2
    need = lib.moe_workspace_size(T, H, I, E, K)
    assert need >= T * K * (H + 2 * I + I + 2 * H)
    assert lib.moe_workspace_size(2 * T, H, I, E, K) > need
    base = [GOOD, GOOD, None, GOOD, GOOD, GOOD, GOOD, T, H, I, E, 1, 1, K, 1, 1, 1.0, GOOD]
    assert f(*base, P(0x100000), need - 1, None) == WORKSPACE
    assert f(*base, None, need, None) == WORKSPACE
    bad_i = list(base)
    bad_i[9] = 48
    assert f(*bad_i, P(0x100000), need, None) == INVALID
    bad_w = list(base)
    bad_w[3] = None
    assert f(*bad_w, P(0x100000), need, None) == INVALID
    # T == 0 is a valid no-op
    assert f(None, None, None, GOOD, GOOD, GOOD, GOOD, 0, H, I, E, 1, 1, K, 1, 1, 1.0, None,
             P(0x100000), lib.moe_workspace_size(0, H, I, E, K), None) == OK


def test_forward_shared_validation(lib):
    """Shared experts: the workspace must cover E + n_shared experts and
    top_k + n_shared slots; n_shared < 0 and top_k + n_shared > 32 are refused
    before any device work."""
    f, fh = lib.moe_forward_shared, lib.moe_forward_shared_host
    T, H, I, E, K = 16, 128, 64, 8, 2
    need = lib.moe_workspace_size(T, H, I, E + 1, K + 1)
    assert need > lib.moe_workspace_size(T, H, I, E, K)

    def base(S):
        return [GOOD, GOOD, None, GOOD, GOOD, GOOD, GOOD, T, H, I, E, S, 1, 1, K, 1, 1, 1.0,
                GOOD]
    ws = P(0x100000)
    assert f(*base(1), ws, lib.moe_workspace_size(T, H, I, E, K), None) == WORKSPACE
    assert f(*base(1), ws, need - 1, None) == WORKSPACE
    assert f(*base(-1), ws, need, None) == INVALID
    assert f(*base(31), ws, 1 << 40, None) == UNSUPPORTED      # top_k + n_shared > 32
    assert fh(*base(1), None, need, None) == WORKSPACE
    assert fh(*base(-1), ws, need, None) == INVALID


def test_block_validation(lib):
    """Block FP8 needs the blocked dimensions to be multiples of 128 (I for
    SiLU*mul, so N = 2I a multiple of 256); refused before any device work."""
    g = lib.moe_grouped_gemm_block
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 256, 192, 4, 0, GOOD, None) == INVALID   # Kd
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 192, 256, 4, 0, GOOD, None) == INVALID   # N
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 384, 256, 4, 1, GOOD, None) == INVALID   # I=192
    assert g(GOOD, GOOD, GOOD, GOOD, GOOD, 64, 256, 256, 2048, 0, GOOD, None) == UNSUPPORTED
    assert lib.moe_act_quant_block(GOOD, 10, 192, GOOD, GOOD, None) == INVALID
    p = lib.moe_permute_quant_block
    need = lib.moe_permute_workspace_size(16, 8, 2)
    assert p(GOOD, GOOD, 16, 160, 8, 2, GOOD, GOOD, GOOD, GOOD, P(0x100000), need,
             None) == INVALID
    assert lib.moe_block_workspace_size(16, 160, 128, 8, 2) == 0
    T, H, I, E, K = 256, 256, 128, 8, 2
    need = lib.moe_block_workspace_size(T, H, I, E, K)
    assert need > lib.moe_workspace_size(T, H, I, E, K)   # per-block scales take more room
    f = lib.moe_forward_block
    base = [GOOD, GOOD, None, GOOD, GOOD, GOOD, GOOD, T, H, I, E, 0, 1, 1, K, 1, 1, 1.0, GOOD]
    assert f(*base, P(0x100000), need - 1, None) == WORKSPACE
    bad = list(base)
    bad[9] = 192  # I not a multiple of 128
    assert f(*bad, P(0x100000), 1 << 40, None) == INVALID
    assert lib.moe_forward_block_host(*bad, P(0x100000), 1 << 40, None) == INVALID


def test_nvfp4_validation(lib):
    """NVFP4 needs K in whole 256-element chunks, N in 128-row tiles, positive
    global scales and a stall stage >= 0 for the timeout test; refused before
    any device work."""
    g = lib.moe_grouped_gemm_nvfp4
    args = lambda **kw: [kw.get("A", GOOD), GOOD, kw.get("ga", 0.5), GOOD, GOOD, GOOD, GOOD,
                         64, kw.get("N", 256), kw.get("Kd", 512), kw.get("E", 4),
                         kw.get("epi", 0), GOOD]
    assert g(*args(Kd=128), None) == INVALID                 # K chunks of 256
    assert g(*args(Kd=384), None) == INVALID
    assert g(*args(N=192), None) == INVALID                  # 128-row tiles
    assert g(*args(ga=0.0), None) == INVALID
    assert g(*args(epi=2), None) == INVALID
    assert g(*args(E=2048), None) == UNSUPPORTED
    assert g(*args(A=ODD), None) == INVALID                  # 16-byte alignment
    t = lib.moe_test_gemm_nvfp4_timeout
    assert t(*args(), -1, None) == INVALID
    assert t(*args(Kd=128), 1, None) == INVALID
    a = lib.moe_act_quant_nvfp4
    assert a(GOOD, 10, 48, 0.5, GOOD, GOOD, None) == INVALID   # I % 32
    assert a(GOOD, 10, 64, 0.0, GOOD, GOOD, None) == INVALID   # g
    assert a(None, 10, 64, 0.5, GOOD, GOOD, None) == INVALID
    p = lib.moe_permute_quant_nvfp4
    need = lib.moe_permute_workspace_size(16, 8, 2)
    perm = lambda H, gs: p(GOOD, GOOD, 16, H, 8, 2, gs, GOOD, GOOD, GOOD, GOOD, P(0x100000),
                           need, None)
    assert perm(48, 0.5) == INVALID                           # H % 32
    assert perm(256, 0.0) == INVALID                          # g
    r = lib.moe_nvfp4_arrange_scales
    assert r(GOOD, 4, 256, 128, 0, GOOD, None) == INVALID      # K chunks of 256
    assert r(GOOD, 4, 192, 256, 0, GOOD, None) == INVALID      # 128-row tiles


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.load()


def test_binding_rejects_host_tensors_before_calling_the_library():
    import torch
    f32 = torch.zeros((4, 8), dtype=torch.float32)
    bf = torch.zeros((4, 64), dtype=torch.bfloat16)
    ids = torch.zeros((4, 2), dtype=torch.int32)
    u8 = torch.zeros((4, 64), dtype=torch.uint8)
    off = torch.zeros(9, dtype=torch.int32)
    calls = [
        lambda: moe.moe_gate(f32, None, 1, 1, 2),
        lambda: moe.moe_permute_quant(bf, ids, 8),
        lambda: moe.moe_grouped_gemm(u8, f32[:, 0].contiguous(), u8.view(1, 4, 64),
                                     torch.ones((1, 4)), off[:2].contiguous()),
        lambda: moe.moe_act_quant(bf),
        lambda: moe.moe_unpermute_sum(bf, ids.view(-1), f32[:, :2].contiguous()),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensors"):
            call()


def test_binding_rejects_undersized_prereorder_buffers():
    """Caller-supplied pre-reorder outputs must match T*K rows (a smaller
    buffer would be written past its end); checked before any library call."""
    import torch
    T, H, K, E = 4, 64, 2, 8
    ok = dict(a_q=torch.zeros((T * K, H), dtype=torch.uint8),
              scale_a=torch.zeros(T * K, dtype=torch.float32),
              src2dst=torch.zeros(T * K, dtype=torch.int32),
              offsets=torch.zeros(E + 1, dtype=torch.int32))
    moe._permute_bufs("f", T, H, K, E, **ok)                     # right sizes: accepted
    moe._permute_bufs("f", T, H, K, E, None, None, None, None)   # the binding allocates
    bad = [("a_q", torch.zeros((T * K - 1, H), dtype=torch.uint8)),
           ("a_q", torch.zeros((T * K, H), dtype=torch.int8)),
           ("scale_a", torch.zeros(T * K - 1, dtype=torch.float32)),
           ("src2dst", torch.zeros(T * K, dtype=torch.int64)),
           ("offsets", torch.zeros(E, dtype=torch.int32))]
    for name, t in bad:
        kw = dict(ok, **{name: t})
        with pytest.raises(ValueError, match=name):
            moe._permute_bufs("f", T, H, K, E, **kw)
    # block scales: one per 128 channels
    kw = dict(ok, scale_a=torch.zeros(T * K * 2, dtype=torch.float32))
    moe._permute_bufs("f", T, 256, K, E, **dict(kw, a_q=torch.zeros((T * K, 256), dtype=torch.uint8)),
                      scales_per_row=2)


def test_binding_rejects_undersized_gemm_buffers():
    """The grouped GEMM wrappers check every scale, offset and output tensor
    against what the kernels read and write, before any library call."""
    import torch
    M, N, E, cols = 10, 256, 4, 128
    ok = dict(scale_a=torch.zeros(M, dtype=torch.float32),
              scale_b=torch.zeros(E * N, dtype=torch.float32),
              offsets=torch.zeros(E + 1, dtype=torch.int32),
              C=torch.zeros((M, cols), dtype=torch.bfloat16), row_amax=None)

    def call(**kw):
        a = dict(ok, **kw)
        moe._gemm_bufs("f", M, N, E, cols, a["scale_a"], M, a["scale_b"], E * N, a["offsets"],
                       a["C"], a["row_amax"])

    call()
    call(row_amax=torch.zeros(M, dtype=torch.float32))
    bad = [("scale_a", torch.zeros(M - 1, dtype=torch.float32)),
           ("scale_b", torch.zeros(E * N, dtype=torch.float16)),
           ("offsets", torch.zeros(E, dtype=torch.int32)),
           ("C", torch.zeros((M, cols - 1), dtype=torch.bfloat16)),
           ("C", torch.zeros((M, cols), dtype=torch.float32)),
           ("row_amax", torch.zeros(M - 1, dtype=torch.float32))]
    for name, t in bad:
        with pytest.raises(ValueError, match=name):
            call(**{name: t})


def _desc(**kw):
    d = dict(quant=moe.QUANT_TOKEN, T=16, H=128, I=64, E=8, n_shared=0, num_groups=1,
             topk_group=1, top_k=2, scoring=0, renormalize=1, routed_scaling_factor=1.0,
             bias=None, w13=0x10000, s13=0x10000, w2=0x10000, s2=0x10000, g13=None, g2=None,
             ga1=0.0, ga2=0.0)
    d.update(kw)
    return moe.MoELayerDesc(**d)


def test_pipeline_workspace_size(lib):
    import ctypes
    assert lib.moe_pipeline_workspace_size(None) == 0
    assert lib.moe_pipeline_workspace_size(ctypes.byref(_desc(quant=7))) == 0
    assert lib.moe_pipeline_workspace_size(ctypes.byref(_desc(E=0))) == 0
    assert lib.moe_pipeline_workspace_size(ctypes.byref(_desc(T=0))) == 0
    d = _desc()
    fw = lib.moe_workspace_size(16, 128, 64, 8, 2)
    slots = 2 * (16 * 128 * 2) + 2 * 512 + 2 * (16 * 128 * 2)   # x, logits (256-aligned), out
    assert lib.moe_pipeline_workspace_size(ctypes.byref(d)) >= fw + slots
    blk = _desc(quant=moe.QUANT_BLOCK, I=128)
    assert lib.moe_pipeline_workspace_size(ctypes.byref(blk)) >= lib.moe_block_workspace_size(
        16, 128, 128, 8, 2)
    assert lib.moe_pipeline_workspace_size(ctypes.byref(_desc(quant=moe.QUANT_BLOCK))) == 0


def test_pipelined_call_rejects_bad_arguments_before_any_device_work(lib):
    import ctypes
    d = _desc()
    need = lib.moe_pipeline_workspace_size(ctypes.byref(d))
    one = (ctypes.c_void_p * 1)(0x20000)
    null1 = (ctypes.c_void_p * 1)(None)
    ws = ctypes.c_void_p(0x100000)
    call = lambda n, x, l, o, w, nb: lib.moe_forward_host_pipelined(  # noqa: E731
        ctypes.byref(d), n, x, l, o, w, nb, None)
    cp = lambda a: ctypes.cast(a, ctypes.c_void_p)  # noqa: E731
    assert lib.moe_forward_host_pipelined(None, 1, cp(one), cp(one), cp(one), ws, need, None) == -1
    assert call(0, cp(one), cp(one), cp(one), ws, need) == -1
    assert call(1, None, cp(one), cp(one), ws, need) == -1
    assert call(1, cp(one), cp(null1), cp(one), ws, need) == -1
    assert call(1, cp(one), cp(one), cp(one), ws, need - 1) == -3
    assert call(1, cp(one), cp(one), cp(one), ctypes.c_void_p(0x100008), need) == -3
    assert call(1, cp(one), cp(one), cp(one), None, need) == -3
    bad = _desc(num_groups=3)   # E % num_groups != 0: the forward's own check
    assert lib.moe_forward_host_pipelined(ctypes.byref(bad), 1, cp(one), cp(one), cp(one), ws,
                                          need, None) == -1
