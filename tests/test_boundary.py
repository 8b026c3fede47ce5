"""The C ABI library: it loads, exports every symbol include/kda.h declares, and
rejects invalid calls on the host before any CUDA work (no GPU needed)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_delta_02_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from chunked_gated_delta_02_gb300._lib import lib as load
    return load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    return sorted({n for n in names if n.startswith("kda_")})


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("kda_fwd", "kda_fwd_workspace_size", "kda_status_string", "kda_get_device_status",
                 "kda_debug_chunk_matrices", "kda_max_chunks", "kda_version"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/kda.h but not exported"


def test_bindings_cover_every_symbol():
    from chunked_gated_delta_02_gb300._lib import SIGNATURES
    assert sorted(SIGNATURES) == declared_functions()


def test_version_and_strings(lib):
    assert lib.kda_version() >= 100
    for code in range(6):
        assert lib.kda_status_string(code)
    assert lib.kda_status_string(99) == b"unknown status"


def test_workspace_size(lib):
    # fixed length: B*ceil(T/64) + N chunk slots per head; per (chunk, head) the 128 x 64 fp16
    # matrix, three 64 x K fp16 operands and K fp32 decays, plus a small header
    ws = lib.kda_fwd_workspace_size(2, 2048, 32, 128, 128, 2)
    per_slot = 128 * 64 * 2 + 3 * 64 * 128 * 2 + 128 * 4
    assert (2 * 32 + 2) * 32 * per_slot <= ws <= (2 * 32 + 2) * 32 * per_slot + 5 * 4096
    assert ws % 256 == 0
    assert lib.kda_fwd_workspace_size(0, 10, 1, 64, 64, 0) == 0       # B < 1
    assert lib.kda_fwd_workspace_size(1, -1, 1, 64, 64, 1) == 0       # T < 0
    assert lib.kda_max_chunks(2, 130, 2) == 2 * 3 + 2
    assert lib.kda_max_chunks(1, 0, 3) == 3


FAKE = 0x10000   # a 256-byte aligned address that is never dereferenced


def _call(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, A_log=FAKE, dt_bias=None, lb=-5.0, scale=0.125,
             init=None, final=None, cu=None, B=1, T=64, H=1, K=64, V=64, N=1, o=FAKE, ws=FAKE,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.kda_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["A_log"], a["dt_bias"], a["lb"],
                       a["scale"], a["init"], a["final"], a["cu"], a["B"], a["T"], a["H"], a["K"], a["V"],
                       a["N"], a["o"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(g=None), 1), (dict(beta=None), 1),
    (dict(A_log=None), 1), (dict(o=None), 1),
    (dict(K=96), 2), (dict(V=32), 2), (dict(K=256), 2),
    (dict(lb=-5.5), 1), (dict(lb=0.5), 1), (dict(lb=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(B=0), 1), (dict(T=-1), 1), (dict(H=0), 1), (dict(N=2), 1),
    (dict(cu=FAKE, B=2, N=2), 1),
    (dict(q=FAKE + 8), 1), (dict(o=FAKE + 4), 1), (dict(beta=FAKE + 1), 1), (dict(init=FAKE + 4), 1),
    (dict(final=FAKE + 8), 1), (dict(cu=FAKE + 2, N=1), 1), (dict(dt_bias=FAKE + 4), 1), (dict(dt_bias=FAKE + 8), 1),
    (dict(ws_bytes=100), 3), (dict(ws=FAKE + 16), 3),
])
def test_host_validation_rejects_without_launch(lib, kw, code):
    assert _call(lib, **kw) == code


def test_null_token_tensors_allowed_only_when_empty(lib):
    assert _call(lib, q=None, T=5) == 1
    assert _call(lib, o=None, T=5) == 1


def test_zero_sequences_is_a_no_op(lib):
    # N = 0 packed sequences: nothing to do, no CUDA call is made
    assert _call(lib, cu=FAKE, N=0, T=0) == 0


def test_debug_wait_timeout_rejects_bad_limits_without_launch(lib):
    assert lib.kda_debug_wait_timeout(0, None) == 1
    assert lib.kda_debug_wait_timeout(-5, None) == 1
    assert lib.kda_debug_wait_timeout(1 << 32, None) == 1


def _call_ex(lib, flags, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, A_log=FAKE, dt_bias=None, lb=-5.0, scale=0.125,
             init=None, final=None, cu=None, B=1, T=64, H=1, K=64, V=64, N=1, o=FAKE, ws=FAKE,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.kda_fwd_ex(a["q"], a["k"], a["v"], a["g"], a["beta"], a["A_log"], a["dt_bias"], a["lb"],
                          a["scale"], a["init"], a["final"], a["cu"], a["B"], a["T"], a["H"], a["K"],
                          a["V"], a["N"], flags, a["o"], a["ws"], a["ws_bytes"], a["stream"], None)


def test_fwd_ex_rejects_unknown_flags_without_launch(lib):
    for flags in (0x40, 0x80, 0x10000, 0x80000000, 0x7F):
        assert _call_ex(lib, flags) == 1
    # context parallelism: KDA_CP_SEGMENTS(n) needs n in [2, 64] and excludes KDA_CP_OFF
    for flags in (1 << 8, 65 << 8, 255 << 8, 0x20 | (4 << 8)):
        assert _call_ex(lib, flags) == 1


def test_workspace_size_with_context_parallel_flags(lib):
    CP_OFF = 0x20
    B, T, H, K, V = 1, 4096, 2, 128, 128
    plain = lib.kda_fwd_workspace_size_ex(B, T, H, K, V, 1, 0, CP_OFF)
    per_seg = H * (2 * V + K) * K * 4          # segment end state + transition, and start state
    for n in (2, 3, 7):
        forced = lib.kda_fwd_workspace_size_ex(B, T, H, K, V, 1, 0, n << 8)
        assert plain + n * per_seg <= forced <= plain + n * per_seg + 512
    # never with cu_seqlens: the forced flag changes nothing there
    assert lib.kda_fwd_workspace_size_ex(B, T, H, K, V, 1, 1, 4 << 8) == plain
    # the default size covers the automatic choice: few heads of a long sequence reserve segments
    assert lib.kda_fwd_workspace_size(B, T, H, K, V, 1) >= plain + 2 * per_seg
    # many heads never use it, and short sequences do not either
    assert lib.kda_fwd_workspace_size(2, 2048, 32, K, V, 2) == lib.kda_fwd_workspace_size_ex(2, 2048, 32, K, V, 2, 0, CP_OFF)
    assert lib.kda_fwd_workspace_size(1, 1000, 1, K, V, 1) == lib.kda_fwd_workspace_size_ex(1, 1000, 1, K, V, 1, 0, CP_OFF)
    assert lib.kda_fwd_workspace_size_ex(B, T, H, K, V, 1, 0, 1 << 8) == 0     # one segment: invalid


def test_plan_needs_a_device_and_valid_arguments(lib):
    import ctypes
    n, bv = ctypes.c_int(-1), ctypes.c_int(-1)
    assert lib.kda_fwd_plan(1, 64, 1, 96, 64, 1, 0, 0, ctypes.byref(n), ctypes.byref(bv)) == 2
    assert lib.kda_fwd_plan(1, 64, 1, 64, 64, 1, 0, 1 << 8, ctypes.byref(n), ctypes.byref(bv)) == 1
    assert lib.kda_fwd_plan(0, 64, 1, 64, 64, 1, 0, 0, ctypes.byref(n), ctypes.byref(bv)) == 1


def test_fwd_ex_variant_alignment_rules(lib):
    GATE_PER_HEAD, BETA_F32 = 0x1, 0x2
    # per-channel gate and dt_bias need 16-byte alignment; per head only their element size
    assert _call_ex(lib, 0, g=FAKE + 2) == 1
    assert _call_ex(lib, GATE_PER_HEAD, g=FAKE + 1) == 1
    assert _call_ex(lib, 0, dt_bias=FAKE + 4) == 1
    assert _call_ex(lib, GATE_PER_HEAD, dt_bias=FAKE + 2) == 1
    # fp32 beta needs 4-byte alignment, bf16 beta 2-byte
    assert _call_ex(lib, BETA_F32, beta=FAKE + 2) == 1
    assert _call_ex(lib, 0, beta=FAKE + 1) == 1
    # the other checks still apply under every flag
    for flags in (0x1, 0x2, 0x4, 0x8, 0x10, 0x1F, 0x20, 4 << 8):
        assert _call_ex(lib, flags, K=96) == 2          # unsupported head dim
        assert _call_ex(lib, flags, lb=-6.0) == 1       # lower bound out of range
        assert _call_ex(lib, flags, init=FAKE + 8) == 1  # state alignment


def test_python_binding_has_no_cpu_path(lib):
    """The binding refuses host tensors instead of computing on the CPU: every step runs in the
    CUDA kernels, and there is no fallback."""
    import torch
    import chunked_gated_delta_02_gb300 as kda
    B, T, H, K = 1, 64, 1, 64
    q = torch.zeros(B, T, H, K, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda.fwd(q, q, q, q, torch.zeros(B, T, H, dtype=torch.bfloat16), torch.zeros(H), None, -5.0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kda.fwd_noalloc(q, q, q, q, torch.zeros(B, T, H, dtype=torch.bfloat16), torch.zeros(H), out=q)


def _meta_args(B=1, T=64, H=2, K=64, V=64):
    """Well-formed arguments on the meta device (no storage): the binding's shape, dtype and
    device checks can run on them without a GPU."""
    import torch
    m = dict(device="meta")
    return dict(q=torch.empty(B, T, H, K, dtype=torch.bfloat16, **m),
                k=torch.empty(B, T, H, K, dtype=torch.bfloat16, **m),
                v=torch.empty(B, T, H, V, dtype=torch.bfloat16, **m),
                g=torch.empty(B, T, H, K, dtype=torch.bfloat16, **m),
                beta=torch.empty(B, T, H, dtype=torch.bfloat16, **m),
                A_log=torch.empty(H, dtype=torch.float32, **m),
                out=torch.empty(B, T, H, V, dtype=torch.bfloat16, **m))


@pytest.mark.parametrize("entry", ["fwd", "fwd_noalloc"])
def test_binding_refuses_each_bad_argument(entry):
    """Every tensor argument of fwd and fwd_noalloc, optional ones included, is checked for device,
    dtype, shape and contiguity before the library is called: a host final_state or a wrong-shape
    out never reaches a kernel."""
    import torch
    import chunked_gated_delta_02_gb300 as kda
    B, T, H, K, V = 1, 64, 2, 64, 64
    fn = getattr(kda, entry)

    def call(**over):
        a = _meta_args(B, T, H, K, V)
        a.update(over)
        extra = {}
        for name in ("dt_bias", "initial_state", "final_state", "cu_seqlens"):
            if name in a:
                extra[name] = a.pop(name)
        if entry == "fwd":
            out = a.pop("out")
            fs = extra.pop("final_state", None)
            return fn(a["q"], a["k"], a["v"], a["g"], a["beta"], a["A_log"], out=out, final_state=fs,
                      output_final_state=fs is not None, **extra)
        return fn(a["q"], a["k"], a["v"], a["g"], a["beta"], a["A_log"], out=a["out"], **extra)

    meta = torch.device("meta")
    with pytest.raises(ValueError, match="final_state must be on"):
        call(final_state=torch.empty(B, H, V, K))                                   # host memory
    with pytest.raises(ValueError, match="out must have shape"):
        call(out=torch.empty(B, T, H, V + 1, dtype=torch.bfloat16, device=meta))
    with pytest.raises(ValueError, match="out must be on"):
        call(out=torch.empty(B, T, H, V, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="final_state must be"):
        call(final_state=torch.empty(B, H, V, K, dtype=torch.float16, device=meta))
    with pytest.raises(ValueError, match="initial_state must have shape"):
        call(initial_state=torch.empty(B, H, V, K + 1, device=meta))
    with pytest.raises(ValueError, match="initial_state must be on"):
        call(initial_state=torch.empty(B, H, V, K))
    with pytest.raises(ValueError, match="dt_bias must hold"):
        call(dt_bias=torch.empty(H * K + 1, device=meta))
    with pytest.raises(TypeError, match="cu_seqlens must be"):
        call(cu_seqlens=torch.empty(2, dtype=torch.int64, device=meta))
    with pytest.raises(ValueError, match="must be contiguous"):
        call(k=torch.empty(B, T, K, H, dtype=torch.bfloat16, device=meta).transpose(2, 3))
    with pytest.raises(TypeError, match="v must be"):
        call(v=torch.empty(B, T, H, V, dtype=torch.float16, device=meta))
    # all well formed, but not on a GPU: refused, there is no CPU path
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()
