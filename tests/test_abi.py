"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import chunked_gated_linear_chunk_gb300 as glc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "glacore.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:size_t|glacore_status|const char \*|int|void)\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("gla_fwd", "gla_bwd", "ssd_fwd", "ssd_bwd", "gla_fwd_workspace_size",
              "glacore_status_string", "glacore_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = glc.load()
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(glc.EXPORTS) <= set(declared_functions())


def test_status_strings_and_version():
    lib = glc.load()
    assert lib.glacore_version() >= 100
    for s in range(8):
        assert lib.glacore_status_string(s)
    assert b"range" in lib.glacore_status_string(glc.ERR_RANGE)
    assert b"unknown" in lib.glacore_status_string(99)


def make_problem(**over):
    p = glc.Problem(B=2, T=100, H=4, Hqk=4, K=128, V=128, dtype=glc.BF16, chunk_size=64, scale=0.1,
                    reserved0=0, q=256, k=512, v=768, g=1024, segment_ids=None, n_seqs=2,
                    initial_state=None, workspace=None, workspace_bytes=0)
    for k, v in over.items():
        setattr(p, k, v)
    return p


BAD = [
    dict(B=0), dict(T=-1), dict(H=0), dict(K=0), dict(V=300), dict(Hqk=3), dict(dtype=7),
    dict(reserved0=1), dict(chunk_size=-64), dict(n_seqs=3), dict(q=None), dict(g=None),
    dict(scale=float("nan")),
]


@pytest.mark.parametrize("over", BAD)
def test_invalid_arguments_rejected_before_launch(over):
    lib = glc.load()
    p = make_problem(**over)
    null = ctypes.c_void_p(0)
    o = ctypes.c_void_p(4096)
    assert lib.gla_fwd(ctypes.byref(p), o, null, null) == glc.ERR_INVALID_ARG
    assert lib.gla_bwd(ctypes.byref(p), o, null, o, o, o, o, null, null) == glc.ERR_INVALID_ARG
    assert lib.gla_fwd_workspace_size(ctypes.byref(p)) == 0


# (problem fields, status of gla_bwd without a workspace): chunk lengths a
# kernel family does not run are UNSUPPORTED; the ones it runs get as far as
# the workspace check (WORKSPACE), before any launch
CHUNKS = [
    (dict(chunk_size=128), glc.ERR_UNSUPPORTED),
    (dict(chunk_size=48), glc.ERR_UNSUPPORTED),
    (dict(chunk_size=64), glc.ERR_WORKSPACE),  # tensor-core kernels
    (dict(chunk_size=0), glc.ERR_WORKSPACE),
    (dict(chunk_size=16), glc.ERR_WORKSPACE),  # CUDA-core kernels on a bf16 problem
    (dict(chunk_size=32), glc.ERR_UNSUPPORTED),  # CUDA-core chunk 32 does not fit K = V = 128
    (dict(dtype=glc.F32, chunk_size=64), glc.ERR_UNSUPPORTED),
    (dict(dtype=glc.F32, K=64, V=64, chunk_size=64), glc.ERR_WORKSPACE),
    (dict(dtype=glc.F32, K=64, V=64, chunk_size=32), glc.ERR_WORKSPACE),
    (dict(dtype=glc.F32, K=64, V=64, chunk_size=16), glc.ERR_WORKSPACE),
    (dict(dtype=glc.F32, K=128, V=64, chunk_size=64), glc.ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("over,status", CHUNKS)
def test_chunk_size_contract(over, status):
    lib = glc.load()
    p = make_problem(**over)
    o = ctypes.c_void_p(4096)
    assert lib.gla_bwd(ctypes.byref(p), o, None, o, o, o, o, None, None) == status
    if status == glc.ERR_WORKSPACE:
        assert lib.gla_bwd_workspace_size(ctypes.byref(p)) > 0


def test_chunk_16_workspace_holds_chunk_states():
    """chunk_size 16 moves a tensor-core problem to the CUDA-core kernels,
    whose backward keeps the fp32 state entering every 16-token chunk."""
    lib = glc.load()
    p = make_problem(chunk_size=16)
    B, T, H, K, V = p.B, p.T, p.H, p.K, p.V
    states = B * ((T + 15) // 16) * H * K * V * 4
    assert lib.gla_bwd_workspace_size(ctypes.byref(p)) >= states


@pytest.mark.parametrize("over", [dict(q_stride=-8), dict(k_stride=4 * 128 - 8), dict(v_stride=100)])
def test_bad_token_strides_rejected(over):
    lib = glc.load()
    p = make_problem(**over)
    o = ctypes.c_void_p(4096)
    assert lib.gla_bwd(ctypes.byref(p), o, None, o, o, o, o, None, None) == glc.ERR_INVALID_ARG
    assert lib.gla_fwd_workspace_size(ctypes.byref(p)) == 0


def test_fused_projection_strides_accepted():
    """q, k, v of one projection [B, T, 3 H K]: each token stride is 3 H K."""
    lib = glc.load()
    p = make_problem(q_stride=3 * 4 * 128, k_stride=3 * 4 * 128, v_stride=3 * 4 * 128)
    o = ctypes.c_void_p(4096)
    assert lib.gla_bwd(ctypes.byref(p), o, None, o, o, o, o, None, None) == glc.ERR_WORKSPACE


def test_shared_qk_heads_keep_per_head_gradients_in_the_workspace():
    """GLA with H / Hqk = 4 on the tensor-core kernels: the backward's
    workspace holds dq and dk per value head (bf16) before the group sum."""
    lib = glc.load()
    p_shared = make_problem(Hqk=1)
    p_own = make_problem(Hqk=4)
    extra = 2 * p_shared.B * p_shared.T * p_shared.H * 128 * 2
    assert lib.gla_bwd_workspace_size(ctypes.byref(p_shared)) >= lib.gla_bwd_workspace_size(ctypes.byref(p_own)) + extra


def test_selftest_wait_rejects_bad_limits():
    lib = glc.load()
    assert lib.glacore_selftest_wait(0, None) == glc.ERR_INVALID_ARG
    assert lib.glacore_selftest_wait(-5, None) == glc.ERR_INVALID_ARG
    assert lib.glacore_selftest_wait((1 << 40) + 1, None) == glc.ERR_INVALID_ARG


def test_missing_outputs_rejected():
    lib = glc.load()
    p = make_problem()
    assert lib.gla_fwd(ctypes.byref(p), None, None, None) == glc.ERR_INVALID_ARG
    o = ctypes.c_void_p(4096)
    assert lib.gla_bwd(ctypes.byref(p), o, None, o, None, o, o, None, None) == glc.ERR_INVALID_ARG


def test_workspace_checked():
    lib = glc.load()
    p = make_problem()
    need = lib.gla_bwd_workspace_size(ctypes.byref(p))
    assert need > 0
    o = ctypes.c_void_p(4096)
    assert lib.gla_bwd(ctypes.byref(p), o, None, o, o, o, o, None, None) == glc.ERR_WORKSPACE
    p.workspace = 4096 + 16  # misaligned
    p.workspace_bytes = need
    assert lib.gla_bwd(ctypes.byref(p), o, None, o, o, o, o, None, None) == glc.ERR_WORKSPACE


def test_segments_need_positive_doc_count():
    lib = glc.load()
    p = make_problem(segment_ids=2048, n_seqs=0)
    assert lib.gla_fwd(ctypes.byref(p), ctypes.c_void_p(4096), None, None) == glc.ERR_INVALID_ARG
    p = make_problem(segment_ids=2048, n_seqs=201)  # more documents than tokens
    assert lib.gla_fwd(ctypes.byref(p), ctypes.c_void_p(4096), None, None) == glc.ERR_INVALID_ARG


def test_empty_problem_is_a_no_op():
    lib = glc.load()
    p = make_problem(T=0, n_seqs=0, q=None, k=None, v=None, g=None)
    assert lib.gla_fwd(ctypes.byref(p), None, None, None) == glc.OK
    assert lib.gla_bwd_workspace_size(ctypes.byref(p)) >= 0


def test_binding_refuses_cpu_tensors():
    import torch

    x = torch.zeros(1, 4, 1, 8)
    with pytest.raises(ValueError):
        glc.gla_fwd(x, x, x, torch.zeros(1, 4, 1, 8))


def test_ssd_forward_needs_no_copies():
    """SSD with one B/C group and V = 64 (workload 3's shape) runs its own
    tensor-core forward on the grouped q / k, the per-head gate and v in
    place: no workspace for plain rows, only the launch order (one int32 per
    document) for a packed batch."""
    lib = glc.load()
    B, T, H, K, V = 4, 4096, 32, 128, 64
    p = make_problem(B=B, T=T, H=H, Hqk=1, K=K, V=V, n_seqs=B, scale=1.0)
    assert lib.ssd_fwd_workspace_size(ctypes.byref(p)) == 0
    packed = make_problem(B=B, T=T, H=H, Hqk=1, K=K, V=V, n_seqs=100, scale=1.0, segment_ids=2048)
    ws = lib.ssd_fwd_workspace_size(ctypes.byref(packed))
    assert 100 * 4 <= ws <= 4096
