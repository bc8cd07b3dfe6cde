"""GB300 (sm_103a) speculative-decoding verification: Python binding.

The work runs in the CUDA kernels of libspec_verify.so behind the C ABI declared
in include/spec_verify.h; this module only checks tensors and marshals pointers
(ctypes).  PyTorch provides device memory and the current stream.  There is no
CPU fallback: if the library is missing, every call raises.

    out_tokens, out_num = verify(target_logits, draft_logits, draft_tokens,
                                 num_draft, uniforms, temperature)

Inputs are CUDA tensors, or page-locked host tensors (``pin_memory()``) that
the kernels read over the host link without a staging copy; outputs are CUDA
tensors.  A page-locked input is read while the kernel runs, after the call has
returned: the binding keeps a reference to it until the launch stream has
passed the call (an event recorded after the launch), so that torch's pinned
memory cache cannot hand the block to another tensor earlier.  The caller must
not change its contents before then.  See include/spec_verify.h for the
operation, layouts and error behaviour.
"""
from __future__ import annotations

import ctypes

from . import _native

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_CUDA = 3

SPEC_F32 = 0
SPEC_BF16 = 1

STATUS_BAD_TOKEN = 1
STATUS_BAD_TEMPERATURE = 2
STATUS_BAD_NUM_DRAFT = 4
STATUS_BAD_LOGITS = 8
STATUS_BAD_TREE = 32

MAX_GAMMA = 16
MAX_TREE_NODES = 256


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = _native.load()
        super().__init__(f"{where}: {lib.spec_status_string(code).decode()} (code {code})")
        self.code = code


def build(force: bool = False) -> str:
    return _native.build(force=force)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must live on {device}, found {t.device}")


def _check_input(t, name, dtype, shape, device):
    """An array the kernels only read: a tensor on ``device``, or a page-locked
    host tensor that the kernels read over the host link (zero copy)."""
    if t.device.type == "cpu":
        _check(t, name, dtype, shape, t.device)
        if t.numel() and not t.is_pinned():  # an empty tensor is never read
            raise ValueError(f"{name}: a host tensor must be page-locked (pin_memory()) for the GPU to read it")
    else:
        _check(t, name, dtype, shape, device)


def _in_ptr(t):
    """Address the kernels use for an input: the CUDA tensor's own, or the
    device alias of a page-locked host tensor (spec_device_pointer)."""
    if t is None or t.is_cuda or t.numel() == 0:
        return _ptr(t)
    out = ctypes.c_void_p()
    rc = _native.load().spec_device_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(out))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_device_pointer")
    return out


def _device_of(*tensors):
    """The CUDA device of the first CUDA tensor given, else the current one."""
    import torch

    for t in tensors:
        if t is not None and t.is_cuda:
            return t.device
    return torch.device("cuda", torch.cuda.current_device())


def _prepare(target, draft, tokens, num_draft, uniforms, temperature, out_tokens, out_num):
    import torch

    if target.dim() != 3:
        raise ValueError("target_logits must be a [B, gamma_max + 1, V] tensor")
    dev = _device_of(target, draft, tokens, num_draft, uniforms, temperature, out_tokens, out_num)
    B, g1, V = target.shape
    gmax = g1 - 1
    code = _dtype_code(target)
    _check_input(target, "target_logits", target.dtype, (B, gmax + 1, V), dev)
    if draft is not None:  # None: point-mass proposals (q_i is 1 at the drafted id)
        _check_input(draft, "draft_logits", target.dtype, (B, gmax, V), dev)
    _check_input(tokens, "draft_tokens", torch.int32, (B, gmax), dev)
    _check_input(num_draft, "num_draft", torch.int32, (B,), dev)
    _check_input(uniforms, "uniforms", torch.float32, (B, gmax + 1), dev)
    _check_input(temperature, "temperature", torch.float32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, gmax + 1), dtype=torch.int32, device=dev)
    if out_num is None:
        out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, gmax + 1), dev)
    _check(out_num, "out_num_accepted", torch.int32, (B,), dev)
    return B, gmax, V, code, out_tokens, out_num


def _status_ptr(t, device):
    """Device pointer of the optional status word: an int32 CUDA tensor on
    ``device`` with at least one element (the kernels OR bits into element 0)."""
    import torch

    if t is None:
        return None
    if t.dtype != torch.int32 or t.device != device or t.numel() < 1 or not t.is_contiguous():
        raise ValueError(f"status must be a contiguous int32 tensor on {device} with at least one element")
    return ctypes.c_void_p(t.data_ptr())


# Page-locked host inputs of launches the stream may not have passed yet:
# (event recorded after the launch, the tensors).  A reference is dropped once
# its event has completed, so torch's pinned-memory cache cannot reuse a block
# that a running kernel still reads.
_held = []


def _hold_host_inputs(tensors, stream, device):
    import torch

    global _held
    host = [t for t in tensors if t is not None and not t.is_cuda and t.numel()]
    if not host and not _held:
        return
    s = torch.cuda.current_stream(device) if stream is None else stream
    with torch.cuda.stream(s):
        if torch.cuda.is_current_stream_capturing():
            # a captured launch reads its inputs at every replay: the caller
            # keeps them for as long as the graph is replayed
            return
    _held = [(ev, ts) for ev, ts in _held if not ev.query()]
    if not host:
        return
    ev = torch.cuda.Event()
    ev.record(s)
    _held.append((ev, host))


def _counter_ptr(t, n, name):
    """Device pointer of an optional int64 CUDA tensor of at least n elements."""
    if t is None:
        return None
    if not t.is_cuda or t.element_size() != 8 or t.numel() < n or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of at least {n} 64-bit integers")
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    import torch

    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


KERNEL_AUTO = 0
KERNEL_REGISTER = 2  # full sweep, register loads
KERNEL_EARLY = 3     # row-ordered early exit: no row after the first rejection is read


def verify(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens=None,
           out_num_accepted=None, status=None, stream=None, cluster_size: int = 0, kernel: int = KERNEL_AUTO,
           counters=None, accept_hist=None):
    """One verification round on the GPU (asynchronous on ``stream``).

    Returns (out_tokens [B, gamma_max+1] int32, out_num_accepted [B] int32).
    ``status``: optional int32 CUDA tensor of one element receiving the
    per-sequence data-problem bits (STATUS_*), OR-ed; zero it first.
    ``cluster_size``: 0 = automatic, else 1 to 16 CTAs per sequence.
    ``kernel``: KERNEL_AUTO, KERNEL_REGISTER or KERNEL_EARLY.
    ``draft_logits=None``: point-mass proposals (a deterministic proposer such
    as ngram_propose): accept iff u < p(x), a rejection samples p without x.
    Inputs may be page-locked host tensors (zero copy; with KERNEL_EARLY only
    the rows up to the first rejection cross the host link); they must stay
    unchanged until the stream has passed the call (the binding keeps them
    alive that long).
    ``counters``: optional uint64 (int64) CUDA tensor [3], += drafted ids,
    accepted ids, verified sequences.  ``accept_hist``: optional int64 CUDA
    tensor [MAX_GAMMA + 1], += 1 at each verified sequence's accepted count.
    """
    B, gmax, V, code, out_tokens, out_num_accepted = _prepare(
        target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, out_tokens, out_num_accepted)
    lib = _native.load()
    args = [_in_ptr(target_logits), _in_ptr(draft_logits), _in_ptr(draft_tokens), _in_ptr(num_draft),
            _in_ptr(uniforms), _in_ptr(temperature), _ptr(out_tokens), _ptr(out_num_accepted), B, gmax, V, code,
            _status_ptr(status, out_tokens.device), _stream_handle(stream, out_tokens.device)]
    if cluster_size or kernel or counters is not None or accept_hist is not None:
        opts = _native.Options(int(cluster_size), int(kernel), _counter_ptr(counters, 3, "counters"),
                               _counter_ptr(accept_hist, MAX_GAMMA + 1, "accept_hist"))
        rc = lib.spec_verify_ex(*args, ctypes.byref(opts))
    else:
        rc = lib.spec_verify(*args)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify")
    _hold_host_inputs((target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature), stream,
                      out_tokens.device)
    return out_tokens, out_num_accepted


def verify_debug(target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, stream=None,
                 cluster_size: int = 0, kernel: int = KERNEL_AUTO):
    """verify() plus the float32 diagnostics of spec_verify_debug (a dict of tensors)."""
    import torch

    B, gmax, V, code, out_tokens, out_num = _prepare(
        target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature, None, None)
    dev = out_tokens.device
    f32 = dict(dtype=torch.float32, device=dev)
    d = {
        "p_hat": torch.empty((B, gmax), **f32),
        "q_hat": torch.empty((B, gmax), **f32),
        "logz_t": torch.empty((B, gmax + 1), **f32),
        "logz_d": torch.empty((B, gmax), **f32),
        "resid_mass": torch.empty((B,), **f32),
        "seq_status": torch.empty((B,), dtype=torch.int32, device=dev),
        "status": torch.zeros((1,), dtype=torch.int32, device=dev),
    }
    lib = _native.load()
    rc = lib.spec_verify_debug(_in_ptr(target_logits), _in_ptr(draft_logits), _in_ptr(draft_tokens),
                               _in_ptr(num_draft), _in_ptr(uniforms), _in_ptr(temperature), _ptr(out_tokens),
                               _ptr(out_num), B, gmax, V,
                               code, _ptr(d["status"]), _stream_handle(stream, dev), _ptr(d["p_hat"]),
                               _ptr(d["q_hat"]), _ptr(d["logz_t"]), _ptr(d["logz_d"]), _ptr(d["resid_mass"]),
                               _ptr(d["seq_status"]),
                               ctypes.byref(_native.Options(int(cluster_size), int(kernel))))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_debug")
    _hold_host_inputs((target_logits, draft_logits, draft_tokens, num_draft, uniforms, temperature), stream, dev)
    d["out_tokens"] = out_tokens
    d["out_num_accepted"] = out_num
    return d


def tree_verify(target_logits, parent, tokens, num_nodes, uniforms, temperature, out_tokens=None,
                out_num_accepted=None, out_path=None, status=None, stream=None, cluster_size: int = 0,
                counters=None, accept_hist=None):
    """One candidate-tree round on the GPU (spec_tree_verify; asynchronous on ``stream``).

    target_logits [B, N, V] (row k: the target after the path to node k);
    parent, tokens [B, N] int32 (node 0 is the root); num_nodes [B] int32;
    uniforms [B, N] float32 (column c tests node c, column 0 drives the final
    sample); temperature [B] float32.  Returns (out_tokens [B, N],
    out_num_accepted [B], out_path [B, N]), int32.
    """
    import torch

    if target_logits.dim() != 3:
        raise ValueError("target_logits must be a [B, N, V] tensor")
    dev = _device_of(target_logits, parent, tokens, num_nodes, uniforms, temperature, out_tokens, out_num_accepted,
                     out_path)
    B, N, V = target_logits.shape
    code = _dtype_code(target_logits)
    _check_input(target_logits, "target_logits", target_logits.dtype, (B, N, V), dev)
    _check_input(parent, "parent", torch.int32, (B, N), dev)
    _check_input(tokens, "tokens", torch.int32, (B, N), dev)
    _check_input(num_nodes, "num_nodes", torch.int32, (B,), dev)
    _check_input(uniforms, "uniforms", torch.float32, (B, N), dev)
    _check_input(temperature, "temperature", torch.float32, (B,), dev)
    i32 = dict(dtype=torch.int32, device=dev)
    out_tokens = torch.empty((B, N), **i32) if out_tokens is None else out_tokens
    out_num_accepted = torch.empty((B,), **i32) if out_num_accepted is None else out_num_accepted
    out_path = torch.empty((B, N), **i32) if out_path is None else out_path
    _check(out_tokens, "out_tokens", torch.int32, (B, N), dev)
    _check(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    _check(out_path, "out_path", torch.int32, (B, N), dev)
    opts = _native.Options(int(cluster_size), 0, _counter_ptr(counters, 3, "counters"),
                           _counter_ptr(accept_hist, MAX_GAMMA + 1, "accept_hist"))
    lib = _native.load()
    rc = lib.spec_tree_verify(_in_ptr(target_logits), _in_ptr(parent), _in_ptr(tokens), _in_ptr(num_nodes),
                              _in_ptr(uniforms), _in_ptr(temperature), _ptr(out_tokens), _ptr(out_num_accepted), _ptr(out_path), B, N, V,
                              code, _status_ptr(status, dev), _stream_handle(stream, dev), ctypes.byref(opts))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_tree_verify")
    _hold_host_inputs((target_logits, parent, tokens, num_nodes, uniforms, temperature), stream, dev)
    return out_tokens, out_num_accepted, out_path


def tree_to_device(tb, device="cuda"):
    """Copy a workloads.TreeBatch (host numpy arrays) to device tensors."""
    import numpy as np
    import torch

    if tb.dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(tb.target).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(tb.target, dtype=np.float32))
    return dict(
        target_logits=t.to(device),
        parent=torch.from_numpy(np.ascontiguousarray(tb.parent, dtype=np.int32)).to(device),
        tokens=torch.from_numpy(np.ascontiguousarray(tb.tokens, dtype=np.int32)).to(device),
        num_nodes=torch.from_numpy(np.ascontiguousarray(tb.num_nodes, dtype=np.int32)).to(device),
        uniforms=torch.from_numpy(np.ascontiguousarray(tb.uniforms, dtype=np.float32)).to(device),
        temperature=torch.from_numpy(np.ascontiguousarray(tb.temperature, dtype=np.float32)).to(device),
    )


def sample(logits, uniforms, temperature, out_tokens=None, status=None, stream=None, cluster_size: int = 0,
           kernel: int = KERNEL_AUTO):
    """One token per row: y_b ~ softmax(logits[b] / T_b) by inverse CDF with
    uniforms[b], or argmax when T_b == 0 (spec_sample).  Draft-side sampling of
    a proposer, or target-only decoding.  Returns out_tokens [B] int32."""
    import torch

    if logits.dim() != 2:
        raise ValueError("logits must be a [B, V] tensor")
    dev = _device_of(logits, uniforms, temperature, out_tokens)
    B, V = logits.shape
    code = _dtype_code(logits)
    _check_input(logits, "logits", logits.dtype, (B, V), dev)
    _check_input(uniforms, "uniforms", torch.float32, (B,), dev)
    _check_input(temperature, "temperature", torch.float32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(out_tokens, "out_tokens", torch.int32, (B,), dev)
    lib = _native.load()
    opts = _native.Options(int(cluster_size), int(kernel))
    rc = lib.spec_sample(_in_ptr(logits), _in_ptr(uniforms), _in_ptr(temperature), _ptr(out_tokens), B, V, code,
                         _status_ptr(status, dev), _stream_handle(stream, dev), ctypes.byref(opts))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_sample")
    _hold_host_inputs((logits, uniforms, temperature), stream, dev)
    return out_tokens


def ngram_propose(context, context_len, min_n: int, max_n: int, gamma_max: int, out_tokens=None, out_num=None,
                  stream=None):
    """Prompt-lookup drafts (spec_ngram_propose): context int32 [B, S] CUDA tensor
    (row b holds context_len[b] tokens), returns (draft_tokens [B, gamma_max],
    num_draft [B]) for spec_verify with draft_logits=None."""
    import torch

    if context.dim() != 2 or context.dtype != torch.int32:
        raise ValueError("context must be an int32 [B, S] tensor")
    dev = _device_of(context, context_len, out_tokens, out_num)
    B = context.shape[0]
    if context.stride(1) != 1:
        raise ValueError("context rows must be contiguous")
    if context.device.type == "cpu" and not context.is_pinned():
        raise ValueError("context: a host tensor must be page-locked (pin_memory()) for the GPU to read it")
    if context.is_cuda and context.device != dev:
        raise ValueError(f"context must live on {dev}, found {context.device}")
    _check_input(context_len, "context_len", torch.int32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma_max), dtype=torch.int32, device=dev)
    if out_num is None:
        out_num = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(out_tokens, "draft_tokens", torch.int32, (B, gamma_max), dev)
    _check(out_num, "num_draft", torch.int32, (B,), dev)
    lib = _native.load()
    rc = lib.spec_ngram_propose(_in_ptr(context), int(context.stride(0)), _in_ptr(context_len), B, int(min_n),
                                int(max_n), int(gamma_max), _ptr(out_tokens), _ptr(out_num),
                                _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_ngram_propose")
    _hold_host_inputs((context, context_len), stream, dev)
    return out_tokens, out_num


def launch_shape(B: int, gamma_max: int, V: int, dtype: str = "bf16"):
    """(cluster size, CTAs, threads per CTA, kernel) the library picks for these
    sizes on the current device; kernel is KERNEL_REGISTER or KERNEL_EARLY."""
    lib = _native.load()
    c, n, t, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = lib.spec_verify_launch_shape(B, gamma_max, V, SPEC_BF16 if dtype == "bf16" else SPEC_F32,
                                      ctypes.byref(c), ctypes.byref(n), ctypes.byref(t), ctypes.byref(k))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_launch_shape")
    return c.value, n.value, t.value, k.value


def to_device(batch, device="cuda"):
    """Copy a workloads.Batch (host numpy arrays) to device tensors, logits in their stored dtype."""
    import numpy as np
    import torch

    if batch.dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(batch.target).view(np.int16)).view(torch.bfloat16)
        d = torch.from_numpy(np.ascontiguousarray(batch.draft).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(batch.target, dtype=np.float32))
        d = torch.from_numpy(np.ascontiguousarray(batch.draft, dtype=np.float32))
    return dict(
        target_logits=t.to(device),
        draft_logits=d.to(device),
        draft_tokens=torch.from_numpy(np.ascontiguousarray(batch.tokens, dtype=np.int32)).to(device),
        num_draft=torch.from_numpy(np.ascontiguousarray(batch.num_draft, dtype=np.int32)).to(device),
        uniforms=torch.from_numpy(np.ascontiguousarray(batch.uniforms, dtype=np.float32)).to(device),
        temperature=torch.from_numpy(np.ascontiguousarray(batch.temperature, dtype=np.float32)).to(device),
    )
