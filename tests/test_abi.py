"""The C-ABI library loads, exports what include/*.h declare, and rejects bad
arguments on the host (no GPU needed: these paths return before any CUDA call).

The calls below pass fake, never-dereferenced device addresses.  They are only
made in a process that sees no GPU, so that even a regression in the checks
could not launch a kernel on them: where this process sees a GPU, the module
runs again in a child process with CUDA_VISIBLE_DEVICES empty and its tests
here are skipped."""
import os
import re
import subprocess
import sys

import pytest

import online_softmax_tiling_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gpu_visible() -> bool:
    if os.environ.get("CUDA_VISIBLE_DEVICES", None) == "":
        return False
    try:
        import torch
        return torch.cuda.is_available()
    except ImportError:
        return False


GPU_VISIBLE = _gpu_visible()


def test_validation_runs_where_no_gpu_is_visible():
    """Where a GPU is visible, run this module's tests in a child that sees none."""
    if not GPU_VISIBLE:
        pytest.skip("no GPU visible: the tests below run in this process")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_abi.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            text = open(os.path.join(inc, h), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if GPU_VISIBLE:
        pytest.skip("run by test_validation_runs_where_no_gpu_is_visible in a child process")
    if not os.path.exists(fa.LIBRARY):
        from online_softmax_tiling_gb300 import build
        build.build()
    return fa.library()


def test_header_declares_the_exports():
    assert _declared() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert fa.fa_version() >= 100
    names = [fa.fa_status_string(s) for s in range(6)]
    assert names == ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED",
                     "FA_ERR_CUDA", "FA_ERR_TIMEOUT"]
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


# Fake, never-dereferenced "device" addresses: every call below fails validation.
A = 0x10000


def _call(**kw):
    args = dict(q=A, k=A + 0x1000, v=A + 0x2000, o=A + 0x3000, lse=A + 0x4000, B=1, H=1, N=128,
                d=64, scale=0.125, causal=0, dtype=fa.FA_FP16, stream=None)
    args.update(kw)
    return fa.fa_fwd(**args)


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(lse=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(d=100), fa.FA_ERR_UNSUPPORTED),   # not a multiple of 8 (16-byte rows)
    (dict(d=264), fa.FA_ERR_UNSUPPORTED),   # wider than the widest kernel
    (dict(d=4), fa.FA_ERR_UNSUPPORTED),
    (dict(d=0), fa.FA_ERR_UNSUPPORTED),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),
])
def test_host_validation(lib, kw, want):
    assert _call(**kw) == want


def test_debug_entry_validates_its_controls(lib):
    base = (A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 1, 1, 128, 64, 0.125, 0,
            fa.FA_FP16, None)
    assert fa.fa_fwd_debug(*base, 3, 1.0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_debug(*base, -1, 1.0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_debug(*base, 0, 0.0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_debug(*base, 0, float("nan")) == fa.FA_ERR_INVALID_ARG


def test_splitkv_workspace_size_and_validation(lib):
    assert fa.fa_splitkv_workspace_size(1, 1, 128, 64, 1) == 0
    need = fa.fa_splitkv_workspace_size(2, 3, 1000, 128, 4)
    S, BH, N, d = 4, 6, 1000, 128
    o_bytes = (4 * S * BH * N * d + 255) // 256 * 256       # fp32 partial O
    assert need == o_bytes + 4 * 2 * S * BH * N              # two fp32 log-sums per row
    base = (A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 2, 3, 1000, 128, 0.1, 0, fa.FA_BF16)
    ws = 0x100000
    assert fa.fa_fwd_splitkv(*base, 33, ws, need, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*base, -1, ws, need, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*base, 4, None, need, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv(*base, 4, ws + 16, need, None) == fa.FA_ERR_MISALIGNED
    assert fa.fa_fwd_splitkv(*base, 4, ws, need - 1, None) == fa.FA_ERR_INVALID_ARG
    assert 1 <= fa.fa_splitkv_num_splits(1, 1, 4096, 64, 0) <= fa.FA_MAX_SPLITS
    assert fa.fa_splitkv_num_splits(64, 64, 4096, 128, 0) == 1
    assert fa.fa_splitkv_num_splits(1, 1, 4096, 100, 0) == 1      # unsupported d: no split


def test_split_heuristic_by_mask(lib):
    """With 152 SMs (GB300; also the count used where no device answers).
    Unmasked d = 128 runs units of two 128-row tiles: 128 of them fill one
    wave, and two waves of halves are no shorter, so no split; 32 blocks are
    split to about one wave.  Causal d = 128 grids whose 256-row blocks fit
    in one wave run one-tile units instead (twice as many, longest first):
    split only while those still fit in one wave, as a causal wave lasts as
    long as its longest unit.  Beyond one wave nothing splits."""
    # with no device visible the library counts GB300's 152 SMs
    assert fa.fa_splitkv_num_splits(1, 8, 4000, 128, 0) == 1      # 128 blocks of 256 rows
    assert fa.fa_splitkv_num_splits(1, 8, 4000, 128, 1) == 1      # 256 one-tile units > 152
    assert fa.fa_splitkv_num_splits(1, 4, 4000, 128, 1) == 2      # 128 one-tile units: halved
    assert fa.fa_splitkv_num_splits(1, 10, 4000, 128, 1) == 1     # 160 blocks > 152
    assert fa.fa_splitkv_num_splits(1, 2, 4096, 128, 0) == 5      # 32 blocks: about one wave
    assert fa.fa_splitkv_num_splits(1, 2, 4096, 128, 1) == 3      # 64 one-tile units
    assert fa.fa_splitkv_num_splits(1, 8, 1024, 128, 1) == 2      # two ranges of 4 key tiles at most
    assert fa.fa_splitkv_num_splits(1, 1, 4096, 64, 0) == 8       # 16 blocks, 8 ranges of 512 keys


def test_calls_without_a_device_return_fa_err_cuda(lib):
    """A valid request on a machine whose CUDA calls fail (here: no device
    visible) comes back as FA_ERR_CUDA from the tensor-map or launch step,
    for every entry point that launches."""
    assert _call() == fa.FA_ERR_CUDA
    assert _call(causal=1, d=256, dtype=fa.FA_BF16) == fa.FA_ERR_CUDA
    base = (A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 1, 1, 128, 64, 0.125, 0,
            fa.FA_FP16, None)
    assert fa.fa_fwd_debug(*base, 2, 1.0) == fa.FA_ERR_CUDA     # the simulated launch failure
    assert fa.fa_fwd_splitkv_noalloc(*base[:-1], 2, None) == fa.FA_ERR_CUDA


def test_noalloc_validates_before_its_size_rule(lib):
    """The no-alloc entry point checks its arguments in the order the others
    do: a request that is both invalid and too large for the array reports
    the invalid argument."""
    B, H, N, d = 8, 16, 4096, 128
    assert fa.fa_splitkv_workspace_size(B, H, N, d, 8) > fa.FA_NOALLOC_SCRATCH_BYTES
    big = (B, H, N, d, 0.1, 0)
    args = (A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000)
    assert fa.fa_fwd_splitkv_noalloc(*args, *big, fa.FA_BF16, 8, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_splitkv_noalloc(None, *args[1:], *big, fa.FA_BF16, 8, None) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv_noalloc(*args, *big, 7, 8, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv_noalloc(*args, B, H, N, d, float("nan"), 0, fa.FA_BF16, 8, None) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv_noalloc(A + 8, *args[1:], *big, fa.FA_BF16, 8, None) == \
        fa.FA_ERR_MISALIGNED
    assert fa.fa_fwd_splitkv_noalloc(*args, B, H, N, 100, 0.1, 0, fa.FA_BF16, 8, None) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_splitkv_noalloc(*args, *big, fa.FA_BF16, 33, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_splitkv_noalloc(*args, *big, fa.FA_BF16, -1, None) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d,width", [(8, 64), (64, 64), (72, 128), (96, 128), (128, 128),
                                     (136, 192), (192, 192), (200, 256), (256, 256)])
def test_splitkv_workspace_uses_the_kernel_width(lib, d, width):
    """Partial O rows are as wide as the kernel that serves d (64, 128, 192 or 256)."""
    S, BH, N = 3, 2, 500
    o_bytes = (4 * S * BH * N * width + 255) // 256 * 256
    assert fa.fa_splitkv_workspace_size(1, 2, N, d, S) == o_bytes + 4 * 2 * S * BH * N


def test_fa_fwd_ex_validation(lib):
    a = fa.fa_fwd_args()
    a.q, a.k, a.v, a.o, a.lse = A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000
    a.B, a.H, a.Nq, a.Nk, a.d = 1, 2, 100, 300, 64
    for f in ("q_stride", "k_stride", "v_stride", "o_stride"):
        getattr(a, f)[:] = [2 * 300 * 64, 300 * 64, 64]
    a.lse_stride[:] = [200, 100]
    a.scale, a.mask, a.dtype, a.num_splits = 0.125, 3, fa.FA_FP16, 1
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_INVALID_ARG          # unknown mask
    a.mask = fa.FA_MASK_CAUSAL_BOTTOM_RIGHT
    a.k_stride[2] = 60                                        # not a multiple of 16 bytes
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_MISALIGNED
    a.k_stride[2] = 64
    a.o_stride[1] = 0
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_MISALIGNED
    a.o_stride[1] = 300 * 64
    a.Nk = 0
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_INVALID_ARG
    a.Nk, a.lse_stride[1] = 300, 0
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_INVALID_ARG
    a.lse_stride[1], a.d = 100, 84
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_UNSUPPORTED
    a.d, a.num_splits, a.workspace = 64, 4, None
    assert fa.fa_fwd_ex(a) == fa.FA_ERR_INVALID_ARG          # split without a workspace


def test_ceiling_probes_validate_arguments(lib):
    import ctypes
    assert lib.fa_ceiling_ex2_rate(None, None) == fa.FA_CEIL_ERR_ARG
    out = ctypes.c_double()
    assert lib.fa_ceiling_l2_read(None, 1 << 20, ctypes.byref(out), None) == fa.FA_CEIL_ERR_ARG
    assert lib.fa_ceiling_l2_read(ctypes.c_void_p(A), 1000, ctypes.byref(out), None) == fa.FA_CEIL_ERR_ARG
    assert lib.fa_ceiling_l2_read(ctypes.c_void_p(A + 8), 1 << 20, ctypes.byref(out), None) == \
        fa.FA_CEIL_ERR_ARG


def test_naive_validation(lib):
    base = (A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, 1, 2, 1000, 64, 0.125, 0, fa.FA_FP16)
    need = fa.fa_naive_workspace_size(1, 2, 1000)
    assert need == 2 * ((2 * 1000 * 1000 * 2 + 255) // 256 * 256)   # S and P, 16-bit each
    ws = 0x100000
    assert fa.fa_naive_fwd(*base, ws, need - 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_naive_fwd(*base, None, need, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_naive_fwd(*base, ws + 16, need, None) == fa.FA_ERR_MISALIGNED
    b = list(base); b[7] = 1001                                     # N not a multiple of 8
    assert fa.fa_naive_fwd(*b, ws, need, None) == fa.FA_ERR_UNSUPPORTED
    b = list(base); b[8] = 96
    assert fa.fa_naive_fwd(*b, ws, need, None) == fa.FA_ERR_UNSUPPORTED


def test_split_choice_counts_keys_from_nk(lib):
    a = fa.fa_fwd_args()
    a.B, a.H, a.Nq, a.Nk, a.d = 1, 8, 1, 262144, 128
    assert fa.fa_splitkv_num_splits_ex(a) > 1                  # decoding: one row, many keys
    a.Nk = 256
    assert fa.fa_splitkv_num_splits_ex(a) == 1                 # too few keys to split
    a.B, a.H, a.Nq, a.Nk = 2, 32, 4096, 4096
    assert fa.fa_splitkv_num_splits_ex(a) == 1                 # the grid already fills the GPU
    assert lib.fa_splitkv_num_splits_ex(None) == 1
