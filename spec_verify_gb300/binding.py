"""Thin Python binding of libsmp (include/smp.h): argument marshalling only.

Every step of the sampler and the verifier runs in the library's CUDA kernels;
PyTorch supplies device memory and the current stream.  If the library has not
been built, loading fails loudly: there is no other implementation to fall
back to.
"""

import ctypes
import os

import numpy as np

from . import build as _build

SMP_F32 = 0
SMP_BF16 = 1

STATUS_NAMES = {0: "SMP_OK", 1: "SMP_ERR_INVALID_ARG", 2: "SMP_ERR_DTYPE", 3: "SMP_ERR_CUDA",
                4: "SMP_ERR_UNSUPPORTED", 5: "SMP_ERR_WORKSPACE"}

ROW_BAD_PARAMS = 1
ROW_NONFINITE = 2
ROW_TIMEOUT = 4
ROW_BAD_DRAFT = 8

# Symbols declared in include/smp.h.
EXPORTS = ("smp_sample", "smp_filter_debug", "smp_sample_processed", "smp_sample_rows", "smp_logit_prepass",
           "smp_beam_topk_workspace_bytes", "smp_beam_topk", "smp_spec_verify_workspace_bytes",
           "smp_spec_verify", "smp_spec_verify_params", "smp_spec_verify_rows", "smp_spec_verify_static",
           "smp_status_string", "smp_last_cuda_error", "smp_abi_version")

STATIC_VERIFY_SCRATCH_BYTES = 1 << 20

# Kernels one verifier call launches (the position kernel, then the resolve kernel).
VERIFY_LAUNCHES = 2

_lib = None


class SmpError(RuntimeError):
    pass


def library_path():
    return _build.LIB


def load():
    """Load libsmp.so (built in-tree by spec_verify_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise SmpError(f"libsmp.so is not built ({path}); run "
                       "`python -m spec_verify_gb300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
    lib.smp_sample.argtypes = [vp, i32, i32, i32, vp, u64, u64, vp, vp, vp, vp]
    lib.smp_sample.restype = i32
    lib.smp_filter_debug.argtypes = [vp, i32, i32, i32, vp, u64, u64, vp, vp, vp, vp, vp, vp]
    lib.smp_filter_debug.restype = i32
    lib.smp_sample_processed.argtypes = [vp, i32, i32, i32, vp, vp, vp, i32, vp, u64, u64, vp, vp, vp, vp]
    lib.smp_sample_processed.restype = i32
    lib.smp_sample_rows.argtypes = [vp, i32, i32, i32, vp, vp, vp, i32, vp, u64, u64, u64, vp, vp, vp, vp]
    lib.smp_sample_rows.restype = i32
    lib.smp_logit_prepass.argtypes = [vp, i32, i32, i32, vp, vp, i32, vp, vp, vp]
    lib.smp_logit_prepass.restype = i32
    lib.smp_beam_topk_workspace_bytes.argtypes = [i32, i32, i32]
    lib.smp_beam_topk_workspace_bytes.restype = sz
    lib.smp_beam_topk.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.smp_beam_topk.restype = i32
    lib.smp_spec_verify_workspace_bytes.argtypes = [i32, i32]
    lib.smp_spec_verify_workspace_bytes.restype = sz
    lib.smp_spec_verify.argtypes = [vp, vp, vp, i32, i32, i32, i32, u64, u64, vp, vp, vp, vp, sz, vp]
    lib.smp_spec_verify.restype = i32
    lib.smp_spec_verify_params.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, u64, u64, vp, vp, vp, vp, vp, sz,
                                           vp]
    lib.smp_spec_verify_params.restype = i32
    lib.smp_spec_verify_rows.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, u64, u64, u64, vp, vp, vp, vp, vp,
                                         sz, vp]
    lib.smp_spec_verify_rows.restype = i32
    lib.smp_spec_verify_static.argtypes = [vp, vp, vp, i32, i32, i32, i32, u64, u64, vp, vp, vp, vp]
    lib.smp_spec_verify_static.restype = i32
    lib.smp_status_string.argtypes = [i32]
    lib.smp_status_string.restype = ctypes.c_char_p
    lib.smp_last_cuda_error.argtypes = []
    lib.smp_last_cuda_error.restype = i32
    lib.smp_abi_version.argtypes = []
    lib.smp_abi_version.restype = i32
    _lib = lib
    return lib


def _check(code):
    if code != 0:
        lib = load()
        msg = lib.smp_status_string(code).decode()
        if code == 3:
            msg += f" (cudaError {lib.smp_last_cuda_error()})"
        raise SmpError(msg)


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return SMP_F32
    if t.dtype == torch.bfloat16:
        return SMP_BF16
    raise SmpError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def params_to_device(params, device):
    """A [B] record array of smp_row_params as a device byte tensor."""
    torch = _torch()
    if isinstance(params, torch.Tensor):
        return params
    arr = np.ascontiguousarray(params)
    return torch.from_numpy(arr.view(np.uint8).copy()).to(device)


def sample(logits, params, seed=0, offset=0, out_ids=None, out_probs=None, status=None, stream=None):
    """smp_sample on a [B, V] float32/bfloat16 CUDA tensor.

    params: record array (spec_verify_gb300.workloads.PARAMS_DTYPE) or a
    device byte tensor holding it.  Returns (ids int32 [B], probs float32 [B],
    status int32 [1]) on the logits' device; status=False passes no status
    word (the call then skips clearing it) and returns None in its place.
    """
    torch = _torch()
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or not logits.is_contiguous():
        raise SmpError("logits must be a contiguous [B, V] CUDA tensor")
    batch, vocab = logits.shape
    dev = logits.device
    prm = params_to_device(params, dev)
    out_ids = out_ids if out_ids is not None else torch.empty(batch, dtype=torch.int32, device=dev)
    out_probs = out_probs if out_probs is not None else torch.empty(batch, dtype=torch.float32, device=dev)
    if status is False:
        status = None
    elif status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_sample(_ptr(logits), batch, vocab, _dtype_code(logits), _ptr(prm), seed, offset,
                          _ptr(out_ids), _ptr(out_probs), _ptr(status), _stream(stream)))
    return out_ids, out_probs, status


def sample_processed(logits, params, seed=0, offset=0, allowed=None, history=None, penalty=None, out_ids=None,
                     out_probs=None, status=None, stream=None):
    """smp_sample_processed: smp_sample after the repetition penalty and the
    constraint mask.  allowed: uint32-valued int32 CUDA tensor [B, ceil(V/32)]
    or None; history: int32 CUDA tensor [B, H] (H <= 64) or None; penalty:
    float32 CUDA tensor [B] or None.  Returns (ids, probs, status)."""
    torch = _torch()
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or not logits.is_contiguous():
        raise SmpError("logits must be a contiguous [B, V] CUDA tensor")
    batch, vocab = logits.shape
    dev = logits.device
    prm = params_to_device(params, dev)
    for t, shape in ((allowed, (batch, (vocab + 31) // 32)), (penalty, (batch,))):
        if t is not None and (tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous()):
            raise SmpError(f"expected a contiguous CUDA tensor of shape {shape}")
    hlen = 0
    if history is not None:
        if history.dim() != 2 or history.shape[0] != batch or history.dtype != torch.int32:
            raise SmpError("history must be an int32 [B, H] CUDA tensor")
        hlen = int(history.shape[1])
    out_ids = out_ids if out_ids is not None else torch.empty(batch, dtype=torch.int32, device=dev)
    out_probs = out_probs if out_probs is not None else torch.empty(batch, dtype=torch.float32, device=dev)
    status = status if status is not None else torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_sample_processed(_ptr(logits), batch, vocab, _dtype_code(logits), _ptr(prm), _ptr(allowed),
                                    _ptr(history), hlen, _ptr(penalty), seed, offset, _ptr(out_ids),
                                    _ptr(out_probs), _ptr(status), _stream(stream)))
    return out_ids, out_probs, status


def sample_rows(logits, params, seed=0, offset=0, row_base=0, allowed=None, history=None, penalty=None,
                out_ids=None, out_probs=None, status=None, stream=None):
    """smp_sample_rows: sample_processed for a part of a larger batch whose
    first row has the global index row_base (the Philox counter of row b is
    row_base + b).  The pre-pass inputs may all be None.  Returns (ids,
    probs, status)."""
    torch = _torch()
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or not logits.is_contiguous():
        raise SmpError("logits must be a contiguous [B, V] CUDA tensor")
    batch, vocab = logits.shape
    dev = logits.device
    prm = params_to_device(params, dev)
    for t, shape in ((allowed, (batch, (vocab + 31) // 32)), (penalty, (batch,))):
        if t is not None and (tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous()):
            raise SmpError(f"expected a contiguous CUDA tensor of shape {shape}")
    hlen = 0
    if history is not None:
        if history.dim() != 2 or history.shape[0] != batch or history.dtype != torch.int32:
            raise SmpError("history must be an int32 [B, H] CUDA tensor")
        hlen = int(history.shape[1])
    out_ids = out_ids if out_ids is not None else torch.empty(batch, dtype=torch.int32, device=dev)
    out_probs = out_probs if out_probs is not None else torch.empty(batch, dtype=torch.float32, device=dev)
    if status is False:
        status = None
    elif status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_sample_rows(_ptr(logits), batch, vocab, _dtype_code(logits), _ptr(prm), _ptr(allowed),
                               _ptr(history), hlen, _ptr(penalty), seed, offset, int(row_base), _ptr(out_ids),
                               _ptr(out_probs), _ptr(status), _stream(stream)))
    return out_ids, out_probs, status


def logit_prepass(logits, allowed=None, history=None, penalty=None, status=None, stream=None):
    """smp_logit_prepass: the repetition penalty and the constraint mask
    written into `logits` (a contiguous [B, V] float32/bfloat16 CUDA tensor)
    in place.  Arguments as for sample_processed.  Returns status."""
    torch = _torch()
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or not logits.is_contiguous():
        raise SmpError("logits must be a contiguous [B, V] CUDA tensor")
    batch, vocab = logits.shape
    dev = logits.device
    for t, shape in ((allowed, (batch, (vocab + 31) // 32)), (penalty, (batch,))):
        if t is not None and (tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous()):
            raise SmpError(f"expected a contiguous CUDA tensor of shape {shape}")
    hlen = 0
    if history is not None:
        if history.dim() != 2 or history.shape[0] != batch or history.dtype != torch.int32:
            raise SmpError("history must be an int32 [B, H] CUDA tensor")
        hlen = int(history.shape[1])
    status = status if status is not None else torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_logit_prepass(_ptr(logits), batch, vocab, _dtype_code(logits), _ptr(allowed), _ptr(history),
                                 hlen, _ptr(penalty), _ptr(status), _stream(stream)))
    return status


def filter_debug(logits, params, seed=0, offset=0, stream=None):
    """smp_filter_debug: (ids, probs, full p~ [B, V], kept [B], status)."""
    torch = _torch()
    lib = load()
    if logits.dim() != 2 or not logits.is_cuda or not logits.is_contiguous():
        raise SmpError("logits must be a contiguous [B, V] CUDA tensor")
    batch, vocab = logits.shape
    dev = logits.device
    prm = params_to_device(params, dev)
    ids = torch.empty(batch, dtype=torch.int32, device=dev)
    probs = torch.empty(batch, dtype=torch.float32, device=dev)
    full = torch.empty(batch, vocab, dtype=torch.float32, device=dev)
    kept = torch.empty(batch, dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_filter_debug(_ptr(logits), batch, vocab, _dtype_code(logits), _ptr(prm), seed, offset,
                                _ptr(ids), _ptr(probs), _ptr(full), _ptr(kept), _ptr(status),
                                _stream(stream)))
    return ids, probs, full, kept, status


def spec_verify_workspace_bytes(batch, k):
    return int(load().smp_spec_verify_workspace_bytes(batch, k))


def _verify_shapes(p_logits, q_logits, draft_ids):
    torch = _torch()
    if p_logits.dim() != 3 or q_logits.dim() != 3 or draft_ids.dim() != 2:
        raise SmpError("expected p [B, K+1, V], q [B, K, V], draft_ids [B, K]")
    batch, k1, vocab = p_logits.shape
    k = k1 - 1
    if tuple(q_logits.shape) != (batch, k, vocab) or tuple(draft_ids.shape) != (batch, k):
        raise SmpError("shape mismatch between p, q and draft_ids")
    if p_logits.dtype != q_logits.dtype or draft_ids.dtype != torch.int32:
        raise SmpError("p and q must share a dtype; draft_ids must be int32")
    for t in (p_logits, q_logits, draft_ids):
        if not t.is_cuda or not t.is_contiguous():
            raise SmpError("inputs must be contiguous CUDA tensors")
    return batch, k, vocab


def _verify_outputs(batch, k, dev, workspace, out_accepted, out_ids, status):
    torch = _torch()
    need = spec_verify_workspace_bytes(batch, k)
    if workspace is None:
        workspace = torch.empty(max(need, 8), dtype=torch.uint8, device=dev)
    out_accepted = out_accepted if out_accepted is not None else torch.empty(batch, dtype=torch.int32, device=dev)
    out_ids = out_ids if out_ids is not None else torch.empty(batch, k + 1, dtype=torch.int32, device=dev)
    status = status if status is not None else torch.empty(1, dtype=torch.int32, device=dev)
    return workspace, out_accepted, out_ids, status


def spec_verify(p_logits, q_logits, draft_ids, seed=0, offset=0, workspace=None, out_accepted=None,
                out_ids=None, status=None, stream=None):
    """smp_spec_verify on p [B, K+1, V], q [B, K, V] and draft ids [B, K] (int32).

    Returns (accepted_len int32 [B], ids int32 [B, K+1], status int32 [1]).
    """
    lib = load()
    batch, k, vocab = _verify_shapes(p_logits, q_logits, draft_ids)
    workspace, out_accepted, out_ids, status = _verify_outputs(batch, k, p_logits.device, workspace,
                                                               out_accepted, out_ids, status)
    _check(lib.smp_spec_verify(_ptr(p_logits), _ptr(q_logits), _ptr(draft_ids), batch, k, vocab,
                               _dtype_code(p_logits), seed, offset, _ptr(out_accepted), _ptr(out_ids),
                               _ptr(status), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out_accepted, out_ids, status


def spec_verify_params(p_logits, q_logits, draft_ids, params, seed=0, offset=0, workspace=None,
                       out_accepted=None, out_ids=None, status=None, stream=None, out_alpha=None):
    """smp_spec_verify_params: spec_verify with per-row knobs (temperature,
    filters, greedy), `params` a [B] record array of smp_row_params or a
    device byte tensor holding it (None: temperature 1 on every row).
    out_alpha: a float32 [B, K] CUDA tensor for the acceptance rates, or None
    (not computed).  Returns (accepted_len, ids, status)."""
    lib = load()
    batch, k, vocab = _verify_shapes(p_logits, q_logits, draft_ids)
    dev = p_logits.device
    prm = params_to_device(params, dev) if params is not None else None
    workspace, out_accepted, out_ids, status = _verify_outputs(batch, k, dev, workspace, out_accepted,
                                                               out_ids, status)
    _check(lib.smp_spec_verify_params(_ptr(p_logits), _ptr(q_logits), _ptr(draft_ids), batch, k, vocab,
                                      _dtype_code(p_logits), _ptr(prm), seed, offset, _ptr(out_accepted),
                                      _ptr(out_ids), _ptr(out_alpha), _ptr(status), _ptr(workspace),
                                      workspace.numel(), _stream(stream)))
    return out_accepted, out_ids, status


def spec_verify_rows(p_logits, q_logits, draft_ids, params=None, seed=0, offset=0, row_base=0, workspace=None,
                     out_accepted=None, out_ids=None, status=None, stream=None, out_alpha=None):
    """smp_spec_verify_rows: spec_verify_params for a part of a larger batch
    whose first row has the global index row_base.  Returns (accepted_len,
    ids, status)."""
    lib = load()
    batch, k, vocab = _verify_shapes(p_logits, q_logits, draft_ids)
    dev = p_logits.device
    prm = params_to_device(params, dev) if params is not None else None
    workspace, out_accepted, out_ids, status = _verify_outputs(batch, k, dev, workspace, out_accepted,
                                                               out_ids, status)
    _check(lib.smp_spec_verify_rows(_ptr(p_logits), _ptr(q_logits), _ptr(draft_ids), batch, k, vocab,
                                    _dtype_code(p_logits), _ptr(prm), seed, offset, int(row_base), _ptr(out_accepted),
                                    _ptr(out_ids), _ptr(out_alpha), _ptr(status), _ptr(workspace),
                                    workspace.numel(), _stream(stream)))
    return out_accepted, out_ids, status


def spec_verify_static(p_logits, q_logits, draft_ids, seed=0, offset=0, out_accepted=None, out_ids=None,
                       status=None, stream=None):
    """smp_spec_verify_static: as spec_verify, with the library's own fixed
    device scratch instead of a workspace (for callers that cannot allocate).
    The outputs must be supplied by the caller if it cannot allocate either."""
    torch = _torch()
    lib = load()
    batch, k1, vocab = p_logits.shape
    k = k1 - 1
    dev = p_logits.device
    out_accepted = out_accepted if out_accepted is not None else torch.empty(batch, dtype=torch.int32, device=dev)
    out_ids = out_ids if out_ids is not None else torch.empty(batch, k + 1, dtype=torch.int32, device=dev)
    status = status if status is not None else torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_spec_verify_static(_ptr(p_logits), _ptr(q_logits), _ptr(draft_ids), batch, k, vocab,
                                      _dtype_code(p_logits), seed, offset, _ptr(out_accepted),
                                      _ptr(out_ids), _ptr(status), _stream(stream)))
    return out_accepted, out_ids, status


def beam_topk(logits, beam_scores, width=None, workspace=None, out_parent=None, out_token=None, out_score=None,
              status=None, stream=None):
    """smp_beam_topk on logits [G, W, V] (float32/bfloat16) and beam_scores
    [G, W] (float64) CUDA tensors; width defaults to W.  Returns (parent
    int32 [G, width], token int32 [G, width], score float64 [G, width],
    status int32 [1])."""
    torch = _torch()
    lib = load()
    if logits.dim() != 3 or not logits.is_cuda or not logits.is_contiguous():
        raise SmpError("logits must be a contiguous [G, W, V] CUDA tensor")
    groups, beams, vocab = logits.shape
    if tuple(beam_scores.shape) != (groups, beams) or beam_scores.dtype != torch.float64 or not beam_scores.is_cuda:
        raise SmpError("beam_scores must be a float64 [G, W] CUDA tensor")
    width = beams if width is None else int(width)
    dev = logits.device
    need = int(lib.smp_beam_topk_workspace_bytes(groups, beams, width))
    if workspace is None:
        workspace = torch.empty(max(need, 8), dtype=torch.uint8, device=dev)
    out_parent = out_parent if out_parent is not None else torch.empty(groups, width, dtype=torch.int32, device=dev)
    out_token = out_token if out_token is not None else torch.empty(groups, width, dtype=torch.int32, device=dev)
    out_score = out_score if out_score is not None else torch.empty(groups, width, dtype=torch.float64, device=dev)
    status = status if status is not None else torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib.smp_beam_topk(_ptr(logits), _ptr(beam_scores), groups, beams, vocab, width, _dtype_code(logits),
                             _ptr(out_parent), _ptr(out_token), _ptr(out_score), _ptr(status), _ptr(workspace),
                             workspace.numel(), _stream(stream)))
    return out_parent, out_token, out_score, status
