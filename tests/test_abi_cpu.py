"""Host-side tests of the C ABI (no GPU): the library builds for sm_103a and
loads, exports every entry point include/*.h declares, sizes scale buffers
like the oracle, and rejects bad arguments before touching the device.  Only
calls that fail argument validation are made, so no fake address is ever
dereferenced or launched on."""
import ctypes
import glob
import os
import re

import pytest

import oracle
import rmsnorm_fp4_quant_gb300 as fq
from rmsnorm_fp4_quant_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fq.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "defined"):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("fp4_add_rmsnorm_quant", "fp4_add_rmsnorm_quant_gs", "fp4_quantize",
                 "fp4_dequant", "fp4_sf_size_bytes", "fp4_launch_shape",
                 "fp4_status_string", "fp4_last_cuda_error", "fp4_gemm_nvfp4_bf16",
                 "fp4_gemm_mxfp4_bf16", "fp4_gemm_nvfp4_gelu_bf16", "fp4_gemm_nvfp4_gelu_nvfp4",
                 "fp4_add_rmsnorm_quant_ex", "fp4_gemm_ex", "fp4_read_device_status"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_library_is_built_for_sm103a(L):
    # the fatbin section of the .so carries an sm_103a cubin; nvcc names the
    # arch in the ELF note, readable as plain bytes
    data = open(fq.lib_path(), "rb").read()
    assert b"sm_103a" in data or b"sm_103" in data


@pytest.mark.parametrize("M", [0, 1, 4, 41, 127, 128, 129, 512, 8192, 32768])
@pytest.mark.parametrize("H", [64, 80, 256, 1536, 5120, 7168, 17408, 32768])
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "e4m3b32"])
def test_sf_size_matches_oracle(L, M, H, fmt):
    f = {"nvfp4": fq.FP4_NVFP4, "mxfp4": fq.FP4_MXFP4, "e4m3b32": fq.FP4_E4M3_B32}[fmt]
    b = oracle.block_size(fmt)
    if H % b:
        assert fq.fp4_sf_size_bytes(M, H, f, fq.FP4_SF_ROWMAJOR) == -1
        return
    assert fq.fp4_sf_size_bytes(M, H, f, fq.FP4_SF_ROWMAJOR) == oracle.sf_size_bytes(M, H, fmt, "rowmajor")
    assert fq.fp4_sf_size_bytes(M, H, f, fq.FP4_SF_SWIZZLED) == oracle.sf_size_bytes(M, H, fmt, "swizzled")
    assert fq.fp4_sf_size_bytes(M, H, f, fq.FP4_SF_BOTH) == oracle.sf_size_bytes(M, H, fmt, "swizzled")


def test_sf_size_rejects_bad_arguments(L):
    assert fq.fp4_sf_size_bytes(-1, 256, 0, 0) == -1
    assert fq.fp4_sf_size_bytes(4, 0, 0, 0) == -1
    assert fq.fp4_sf_size_bytes(4, 256, 7, 0) == -1
    assert fq.fp4_sf_size_bytes(4, 256, 0, 9) == -1


def test_status_strings(L):
    for s in range(6):
        assert fq.fp4_status_string(s) and fq.fp4_status_string(s) != "unknown status"
    assert "timeout" in fq.fp4_status_string(fq.FP4_ERR_TIMEOUT)
    assert fq.fp4_status_string(99) == "unknown status"


def test_status_codes_match_the_header(L):
    text = open(os.path.join(ROOT, "include", "fp4q.h")).read()
    for name in ("FP4_OK", "FP4_ERR_INVALID_ARG", "FP4_ERR_UNSUPPORTED_SHAPE",
                 "FP4_ERR_MISALIGNED", "FP4_ERR_CUDA", "FP4_ERR_TIMEOUT", "FP4_EPI_BF16",
                 "FP4_EPI_GELU_BF16", "FP4_EPI_GELU_NVFP4"):
        m = re.search(rf"\b{name}\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == getattr(fq, name), name


def test_read_device_status_rejects_bad_pointers(L):
    # rejected before the stream or the pointer is touched
    assert fq.fp4_read_device_status(0, 0) == fq.FP4_ERR_INVALID_ARG
    assert fq.fp4_read_device_status(A + 2, 0) == fq.FP4_ERR_INVALID_ARG


# Fake, never-dereferenced addresses: every call below must fail validation.
A = 0x7F0000000000           # 4 KiB-aligned
B = A + (1 << 32)
W = A + (2 << 32)
P = A + (3 << 32)
S = A + (4 << 32)
S2 = A + (5 << 32)


def _call(x=A, r=B, w=W, eps=1e-6, M=4, H=256, dt=0, f=0, lay=0, p=P, s=S, s2=0):
    return fq.fp4_add_rmsnorm_quant(x, r, w, eps, M, H, dt, f, lay, p, s, s2, 0)


@pytest.mark.parametrize("kwargs,status", [
    (dict(dt=2), 1), (dict(f=3), 1), (dict(lay=5), 1), (dict(M=-1), 1), (dict(H=0), 1),
    (dict(H=80, f=2), 2),
    (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1),
    (dict(H=40), 2), (dict(H=48), 2), (dict(H=80, f=1), 2), (dict(H=262144 + 16), 2),
    (dict(x=0), 1), (dict(r=0), 1), (dict(w=0), 1), (dict(p=0), 1), (dict(s=0), 1),
    (dict(lay=2, s2=0), 1),
    (dict(x=A + 16), 3), (dict(r=B + 8), 3), (dict(w=W + 2), 3), (dict(p=P + 4), 3),
    (dict(r=A + 512), 1),                    # input and residual overlap
    (dict(p=B + 64), 1),                     # packed inside the residual
    (dict(s=P + 16), 1),                     # scales inside the packed output
    (dict(lay=1, s=S + 2), 3),               # tiled scales need 4-byte alignment
])
def test_fused_validation(L, kwargs, status):
    assert _call(**kwargs) == status


def test_m_zero_is_a_no_op(L):
    # nothing is launched and no pointer is looked at
    assert _call(M=0, x=0, r=0, w=0, p=0, s=0) == 0


@pytest.mark.parametrize("args,status", [
    ((P, S, 4, 256, 2, 0, 0, 0), 1), ((P, S, 4, 256, 0, 2, 0, 0), 1), ((P, S, -1, 256, 0, 0, 0, 0), 1),
    ((P, S, 4, 40, 0, 0, 0, 0), 2), ((0, S, 4, 256, 0, 0, A, 0), 1), ((P + 4, S, 4, 256, 0, 0, A, 0), 3),
    ((P, S, 4, 256, 0, 0, A + 8, 0), 3), ((0, 0, 0, 256, 0, 0, 0, 0), 0),
])
def test_dequant_validation(L, args, status):
    assert fq.fp4_dequant(*args) == status


def test_tensor_api_refuses_cpu_tensors(L):
    import torch
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fq.add_rmsnorm_fp4quant(x, x.clone(), torch.ones(256, dtype=torch.bfloat16))


@pytest.mark.parametrize("kwargs,status", [
    (dict(gs=A + 2), 3),            # global scale must be 4-byte aligned
    (dict(dt=5), 1), (dict(H=40), 2),
])
def test_fused_gs_validation(L, kwargs, status):
    a = dict(x=A, r=B, w=W, gs=0, eps=1e-6, M=4, H=256, dt=0, f=0, lay=0, p=P, s=S, s2=0)
    a.update(kwargs)
    st = fq.fp4_add_rmsnorm_quant_gs(a["x"], a["r"], a["w"], a["gs"], a["eps"], a["M"], a["H"],
                                     a["dt"], a["f"], a["lay"], a["p"], a["s"], a["s2"], 0)
    assert st == status


@pytest.mark.parametrize("kwargs,status", [
    (dict(dt=3), 1), (dict(f=4), 1), (dict(lay=3), 1), (dict(M=-2), 1), (dict(H=24), 2),
    (dict(H=48, f=1), 2), (dict(x=0), 1), (dict(p=0), 1), (dict(s=0), 1), (dict(x=A + 8), 3),
    (dict(gs=W + 1), 3), (dict(p=P + 2), 3), (dict(lay=1, s=S + 1), 3), (dict(p=A + 256), 1),
    (dict(M=0, x=0, p=0, s=0), 0),
])
def test_quantize_validation(L, kwargs, status):
    a = dict(x=A, gs=0, M=4, H=256, dt=0, f=0, lay=0, p=P, s=S, s2=0)
    a.update(kwargs)
    st = fq.fp4_quantize(a["x"], a["gs"], a["M"], a["H"], a["dt"], a["f"], a["lay"], a["p"],
                         a["s"], a["s2"], 0, 0)
    assert st == status


@pytest.mark.parametrize("kwargs,status", [
    (dict(xs=100), 1),                 # row stride below H
    (dict(rs=200), 1),
    (dict(xs=264), 3),                 # rows would not start 32-byte aligned
    (dict(rs=257 * 16 + 8), 3),
    (dict(y=A + (7 << 32) + 16), 3),   # y must be 32-byte aligned
    (dict(y=B + 64), 1),               # y inside the residual
    (dict(y=P + 32), 1),               # y over the packed output
    (dict(xs=512, r=A + 512), 1),      # strided input overlapping the residual
    (dict(st=S2 + 2), 3),              # status word must be 4-byte aligned
    (dict(st=P + 64), 1),              # status word inside the packed output
    (dict(st=A + 64), 1),              # status word inside the input
    (dict(lay=2, s2=P + 16), 1),       # row-major scales of "both" over the packed output
    (dict(lay=2, s2=B + 32), 1),       # ... over the residual
    (dict(lay=2, s2=A), 1),            # ... over the input
    (dict(lay=2, s2=S + 4), 1),        # ... over the tiled scales
    (dict(p=A + 128), 1),              # packed output inside the input
    (dict(p=W), 1),                    # packed output over the weight
    (dict(s=W + 32), 1),               # scales over the weight
    (dict(y=W), 1),                    # y over the weight
    (dict(gs=P + 4), 1),               # global scale read from the packed output
])
def test_fused_ex_validation(L, kwargs, status):
    a = dict(x=A, xs=0, r=B, rs=0, w=W, gs=0, eps=1e-6, M=4, H=256, dt=0, f=0, lay=0, p=P, s=S,
             s2=0, y=0, st=0, pdl=0)
    a.update(kwargs)
    st = fq.fp4_add_rmsnorm_quant_ex(a["x"], a["xs"], a["r"], a["rs"], a["w"], a["gs"], a["eps"],
                                     a["M"], a["H"], a["dt"], a["f"], a["lay"], a["p"], a["s"],
                                     a["s2"], a["y"], a["st"], a["pdl"], 0)
    assert st == status


@pytest.mark.parametrize("kwargs,status", [
    (dict(p=A + 256), 1),              # packed output inside the input
    (dict(lay=2, s2=P + 8), 1),        # row-major scales over the packed output
    (dict(lay=2, s2=S), 1),            # row-major scales over the tiled ones
    (dict(lay=2, s2=A + 64), 1),       # row-major scales inside the input
    (dict(gs=P), 1),                   # global scale read from the packed output
])
def test_quantize_overlap_validation(L, kwargs, status):
    a = dict(x=A, gs=0, M=4, H=256, dt=0, f=0, lay=0, p=P, s=S, s2=0)
    a.update(kwargs)
    st = fq.fp4_quantize(a["x"], a["gs"], a["M"], a["H"], a["dt"], a["f"], a["lay"], a["p"],
                         a["s"], a["s2"], 0, 0)
    assert st == status


G_OUT = A + (6 << 32)


@pytest.mark.parametrize("kwargs,status", [
    (dict(M=-1), 1), (dict(N=-1), 1), (dict(K=0), 1),
    (dict(K=48), 2),                   # K not a multiple of 32
    (dict(K=16), 2),
    (dict(N=20), 2),                   # N not a multiple of 8
    (dict(K=1 << 31), 2),
    (dict(a=0), 1), (dict(b=0), 1), (dict(sfa=0), 1), (dict(sfb=0), 1), (dict(out=0), 1),
    (dict(a=A + 8), 3), (dict(sfb=S + 4), 3), (dict(out=G_OUT + 2), 3), (dict(bias=W + 8), 3),
    (dict(residual=B + 8), 3),
    (dict(out=A + 1024), 1),           # output over A
    (dict(out=S + 512), 1),            # output over the scales of A
    (dict(bias=G_OUT + 64), 1),        # bias inside the output
    (dict(residual=G_OUT + 64), 1),    # residual partly over the output
    (dict(M=0, a=0, b=0, out=0), 0),   # empty: nothing launched
    (dict(N=0), 0),
    (dict(variant=5), 1), (dict(variant=-2), 1),
    (dict(pdl=3), 1), (dict(pdl=-1), 1),          # 0, 1 or 2 (static weights)
])
def test_gemm_validation(L, kwargs, status):
    a = dict(a=A, b=B, sfa=S, sfb=S2, alpha=1.0, bias=0, residual=0, M=256, N=256, K=512,
             out=G_OUT, variant=-1, pdl=0)
    a.update(kwargs)
    st = fq.fp4_gemm_nvfp4_bf16(a["a"], a["b"], a["sfa"], a["sfb"], a["alpha"], a["bias"],
                                a["residual"], a["M"], a["N"], a["K"], a["out"], a["variant"],
                                a["pdl"], 0)
    assert st == status


@pytest.mark.parametrize("kwargs,status", [
    (dict(fmt=2), 1), (dict(fmt=7), 1),          # E4M3-B32 operands, bad enum
    (dict(epi=3), 1), (dict(epi=-1), 1),
    (dict(epi=2, fmt=1), 1),                     # NVFP4 output takes NVFP4 operands only
    (dict(epi=1, residual=B + (1 << 20)), 1),    # GELU takes no residual
    (dict(epi=2, residual=B + (1 << 20)), 1),
    (dict(st=S2 + 1), 3),                        # status word alignment
    (dict(st=G_OUT + 256), 1),                   # status word inside the output
    (dict(st=A + 4), 1),                         # ... inside A
    (dict(epi=2, out=0, p=P, s=G_OUT, st=P + 16), 1),   # ... inside the packed output
    (dict(K=48), 2), (dict(variant=7), 1), (dict(pdl=3), 1),
    (dict(M=0, a=0, b=0, out=0), 0),
])
def test_gemm_ex_validation(L, kwargs, status):
    a = dict(a=A, b=B, sfa=S, sfb=S2, fmt=0, epi=0, alpha=1.0, bias=0, residual=0, M=256, N=256,
             K=512, out=G_OUT, p=0, s=0, variant=-1, pdl=0, st=0)
    a.update(kwargs)
    st = fq.fp4_gemm_ex(a["a"], a["b"], a["sfa"], a["sfb"], a["fmt"], a["epi"], a["alpha"],
                        a["bias"], a["residual"], a["M"], a["N"], a["K"], a["out"], a["p"],
                        a["s"], a["variant"], a["pdl"], a["st"], 0)
    assert st == status


def test_default_build_has_no_debug_knobs(L):
    assert L.fp4_debug_build() == 0
    assert fq.fp4_debug_configure(1000, 0, 1, 0, 0, 0) == fq.FP4_ERR_INVALID_ARG


@pytest.fixture(scope="module")
def D(L):
    fbuild.build(debug=True)
    return fq.debug_lib()


def test_debug_build_exports_the_same_entry_points(D):
    assert D.fp4_debug_build() == 1
    for name in _declared_functions():
        assert ctypes.cast(getattr(D, name), ctypes.c_void_p).value, name


@pytest.mark.parametrize("args,status", [
    ((2_000_000_000, 0, 0, -1, -1, 0), 0),
    ((20_000, 1, 2, 0, 1, A), 0),
    ((0, 0, 0, -1, -1, 0), 1),             # the wait limit must be positive
    ((1000, -1, 0, -1, -1, 0), 1),         # negative shrink
    ((1000, 0, 3, 0, 0, 0), 1),            # no kernel 3
    ((1000, 0, 1, 0, 0, A + 2), 3),        # counter alignment
])
def test_debug_configure_validation(D, args, status):
    """Host only: the knobs are stored, nothing is launched or dereferenced."""
    try:
        assert D.fp4_debug_configure(*args) == status
    finally:
        D.fp4_debug_configure(2_000_000_000, 0, 0, -1, -1, None)


def test_library_exports_only_the_declared_entry_points(L):
    """The library is built with hidden visibility: its dynamic symbol table
    holds exactly the functions include/*.h declares (no internal C++ symbols)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", fq.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(_declared_functions())


@pytest.mark.parametrize("kwargs,status", [
    (dict(variant=5), 1),
    (dict(K=80), 2), (dict(a=0), 1), (dict(sfa=S + 8), 3),   # K not a multiple of 32
    (dict(out=S + 256), 1),                         # output over the MXFP4 scales of A
    (dict(M=0, a=0), 0),
])
def test_gemm_mxfp4_validation(L, kwargs, status):
    a = dict(a=A, b=B, sfa=S, sfb=S2, alpha=1.0, bias=0, residual=0, M=256, N=256, K=512,
             out=G_OUT, variant=-1, pdl=0)
    a.update(kwargs)
    st = fq.fp4_gemm_mxfp4_bf16(a["a"], a["b"], a["sfa"], a["sfb"], a["alpha"], a["bias"],
                                a["residual"], a["M"], a["N"], a["K"], a["out"], a["variant"],
                                a["pdl"], 0)
    assert st == status


@pytest.mark.parametrize("kwargs,status", [
    (dict(variant=4), 1),                 # split K cannot quantize 16-wide blocks
    (dict(N=264), 2),                     # N not a multiple of 16
    (dict(p=0), 1), (dict(s=0), 1),
    (dict(p=A + 64), 1),                  # packed output over A
    (dict(s=P + 128), 1),                 # scales over the packed output
    (dict(p=P + 8), 3),
    (dict(M=0, a=0, p=0, s=0), 0),
])
def test_gemm_gelu_nvfp4_validation(L, kwargs, status):
    a = dict(a=A, b=B, sfa=S, sfb=S2, alpha=1.0, bias=0, M=256, N=256, K=512, p=P,
             s=G_OUT, variant=-1, pdl=0)
    a.update(kwargs)
    st = fq.fp4_gemm_nvfp4_gelu_nvfp4(a["a"], a["b"], a["sfa"], a["sfb"], a["alpha"], a["bias"],
                                      a["M"], a["N"], a["K"], a["p"], a["s"], a["variant"],
                                      a["pdl"], 0)
    assert st == status


def test_gemm_variant_query(L):
    """The schedule query: host only (152 SMs without a device); a given
    variant comes back as given, rejected sizes give -1."""
    import rmsnorm_fp4_quant_gb300 as fq
    v = fq.fp4_gemm_variant
    assert v(8192, 7168, 7168)["variant"] == 3                       # many tiles, NVFP4
    assert v(8192, 7168, 7168)["kernel"] == "gemm_nvfp4_persistent_kernel"
    assert v(8192, 7168, 7168, fmt=1)["variant"] == 3                # MXFP4 as well
    assert v(41, 1536, 6144)["split_k"]                              # few tiles, long K
    assert v(41, 4608, 1536)["variant"] == 0                         # few tiles, 6 K blocks
    assert v(8192, 7168, 7168, fp4_out=True)["variant"] == 3
    assert v(41, 1536, 6144, fp4_out=True)["variant"] == 0           # no split for FP4 output
    assert v(256, 256, 512, variant=3)["variant"] == 3
    assert L.fp4_gemm_variant(256, 256, 240, 0, 0, -1) == -1         # K % 32
    assert L.fp4_gemm_variant(256, 256, 32, 0, 0, -1) >= 0           # one half K step
    assert L.fp4_gemm_variant(41, 520, 288, 1, 0, -1) >= 0           # ragged last K block
    assert L.fp4_gemm_variant(256, 256, 16, 0, 0, -1) == -1
    assert L.fp4_gemm_variant(256, 256, 512, 1, 0, 2) == 2           # MXFP4 persistent
    assert L.fp4_gemm_variant(256, 264, 512, 0, 1, -1) == -1         # FP4 output: N % 16
    assert L.fp4_gemm_variant(256, 256, 512, 2, 0, -1) == -1         # E4M3-B32 operands


def _launch_shape_cases():
    widths = sorted({64, 80, 96, 208, 256, 1536, 2080, 4096, 5120, 6144, 7168, 8224, 12288,
                     16384, 17408} | {16 * k for k in range(4, 129, 7)})
    for H in widths:
        for M in (1, 3, 41, 128, 129, 512, 5000, 32768):
            for fmt in (0, 1, 2):
                yield M, H, fmt


def test_launch_shape_invariants(L):
    """Host-side choice of the fused launch (fp4_launch_shape, 152 SMs without
    a device), over widths up to the register-resident limit, batch sizes and
    formats: every chunk of a row has a thread, thread counts are whole warps
    within the instance's limit, a cluster splits a row evenly (on 32-element
    blocks for the 32-blocks formats), and the grid covers every row the
    call writes (tiled layouts include the padding rows)."""
    import rmsnorm_fp4_quant_gb300 as fq
    checked = 0
    for M, H, fmt in _launch_shape_cases():
        if H % (16 if fmt == 0 else 32):
            continue
        for lay in (0, 1):
            s = fq.fp4_launch_shape(M, H, 0, fmt, lay)
            nchunk = H // 16
            rows = M if lay == 0 else (M + 127) // 128 * 128
            cpt, tpr, R, C = (s["chunks_per_thread"], s["threads_per_slice"],
                              s["slices_per_cta"], s["cluster"])
            assert 1 <= cpt <= 4 and tpr >= 2 and R >= 1, (M, H, s)
            assert s["threads_per_cta"] == tpr * R and s["threads_per_cta"] % 32 == 0, (M, H, s)
            assert s["threads_per_cta"] <= (1024 if cpt == 1 else 512), (M, H, s)
            assert C in (1, 2, 4, 8) and nchunk % C == 0, (M, H, s)
            if fmt != 0:
                assert (nchunk // C) % 2 == 0, (M, H, s)      # whole 32-element blocks
            assert tpr * cpt >= nchunk // C, (M, H, s)          # every chunk has a thread
            if s["kernel"] == "fused_direct_kernel":
                assert s["stages"] == 0
                if C > 1:
                    assert R == 1 and s["ctas"] == rows * C, (M, H, s)
                else:
                    assert s["ctas"] * R >= rows > (s["ctas"] - 1) * R, (M, H, s)
            else:
                assert s["stages"] >= 1 and 1 <= s["ctas"], (M, H, s)
            checked += 1
    assert checked > 500
