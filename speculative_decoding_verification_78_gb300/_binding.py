"""ctypes binding of libspec_verify.so: the C entry points under the same names.

Argument marshalling only: every step of the verify path runs in the library's CUDA kernels.
torch is used for device memory and streams. There is no fallback: when the library is
missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libspec_verify.so")
# the same kernels compiled with SPEC_CHECKED: computed indices range-checked (SPEC_ERR_CHECK)
CHECKED_LIB_PATH = os.path.join(PKG, "libspec_verify_checked.so")

SPEC_F32, SPEC_BF16 = 0, 1
SPEC_OK = 0
SPEC_ERR_NULL, SPEC_ERR_SHAPE, SPEC_ERR_TEMP, SPEC_ERR_DTYPE = -1, -2, -3, -4
SPEC_ERR_WORKSPACE, SPEC_ERR_ALIGN, SPEC_ERR_LAUNCH = -5, -6, -7
SPEC_ERR_NONFINITE, SPEC_ERR_TOKEN, SPEC_ERR_PARENT, SPEC_ERR_CHECK = -20, -21, -22, -24
SPEC_ERR_TIMEOUT = -23
SPEC_MAX_V, SPEC_MAX_GAMMA, SPEC_MAX_NODES = 1 << 20, 255, 1024
SPEC_LMHEAD_MAX_V = 1 << 19

# every symbol include/spec_verify.h declares
EXPORTS = ("spec_workspace_bytes", "spec_workspace_init", "spec_verify_chain",
           "spec_verify_tree", "spec_verify_tree_sample", "spec_lmhead_workspace_bytes",
           "spec_verify_chain_lmhead", "spec_probs", "spec_status_string",
           "spec_last_cuda_error", "spec_cuda_error_string",
           "spec_launch_shape", "spec_verify_chain_static", "spec_sample", "spec_topk",
           "spec_tree_mask", "spec_selftest_bounded_wait")
SPEC_MAX_TOPK = 16
SPEC_STATIC_SCRATCH_BYTES = 4 << 20
SPEC_CALL_CHAIN, SPEC_CALL_TREE, SPEC_CALL_PROBS = 0, 1, 2

_lock = threading.Lock()
_lib = None
_checked_lib = None


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {spec_status_string(code)} ({code})"
        if code == SPEC_ERR_LAUNCH:
            ce = spec_last_cuda_error()
            if ce:
                msg += f"; CUDA error {ce}: {spec_cuda_error_string(ce)}"
        super().__init__(msg)


def load_library(checked: bool = False):
    """Loads libspec_verify.so (built in-tree by __graft_entry__.build()), or with
    checked=True its checked build libspec_verify_checked.so."""
    global _lib, _checked_lib
    with _lock:
        if (_checked_lib if checked else _lib) is not None:
            return _checked_lib if checked else _lib
        path = CHECKED_LIB_PATH if checked else LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.spec_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.spec_workspace_bytes.restype = sz
        lib.spec_workspace_init.argtypes = [vp, sz, vp]
        lib.spec_workspace_init.restype = i32
        lib.spec_verify_chain.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, f32, vp, vp, vp,
                                          vp, sz, vp]
        lib.spec_verify_chain.restype = i32
        lib.spec_verify_tree.argtypes = [vp, i32, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz,
                                         vp]
        lib.spec_verify_tree.restype = i32
        lib.spec_verify_tree_sample.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, f32,
                                                vp, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_tree_sample.restype = i32
        lib.spec_lmhead_workspace_bytes.argtypes = [i32, i32, i32]
        lib.spec_lmhead_workspace_bytes.restype = sz
        lib.spec_verify_chain_lmhead.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, i32, i32, i32,
                                                 f32, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.spec_verify_chain_lmhead.restype = i32
        lib.spec_probs.argtypes = [vp, i32, i32, i32, f32, vp, vp, vp, sz, vp]
        lib.spec_probs.restype = i32
        lib.spec_status_string.argtypes = [i32]
        lib.spec_status_string.restype = ctypes.c_char_p
        lib.spec_last_cuda_error.argtypes = []
        lib.spec_last_cuda_error.restype = i32
        lib.spec_cuda_error_string.argtypes = [i32]
        lib.spec_cuda_error_string.restype = ctypes.c_char_p
        lib.spec_launch_shape.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp]
        lib.spec_launch_shape.restype = i32
        lib.spec_verify_chain_static.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, f32, vp, vp,
                                                 vp, vp]
        lib.spec_verify_chain_static.restype = i32
        lib.spec_sample.argtypes = [vp, i32, i32, i32, f32, vp, vp, vp, vp, sz, vp]
        lib.spec_sample.restype = i32
        lib.spec_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, sz, vp]
        lib.spec_topk.restype = i32
        lib.spec_tree_mask.argtypes = [vp, i32, i32, vp, vp, vp]
        lib.spec_tree_mask.restype = i32
        lib.spec_selftest_bounded_wait.argtypes = [vp, ctypes.c_double, vp]
        lib.spec_selftest_bounded_wait.restype = i32
        if checked:
            _checked_lib = lib
        else:
            _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling helpers

def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t)}")
    if t.numel() and not t.is_cuda:
        raise ValueError("device tensor expected (the library takes device pointers)")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def dtype_flag(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype in (torch.bfloat16, torch.int16) or str(t.dtype) == "torch.uint16":
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16 (got {t.dtype})")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _expect(t, name, numel, dtypes):
    """Raises ValueError / TypeError unless tensor t (when given) holds `numel` elements of one
    of `dtypes`: the library reads and writes exactly that many elements behind each pointer."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {' or '.join(map(str, dtypes))}")
    if t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements ({tuple(t.shape)}), expected {numel}")


def _chain_shape_check(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                       accept_len, out_tokens, status):
    """(B, gamma, V) of a chain call, after checking every operand against them: the draft
    logits [B, gamma, V] of the target's dtype, int32 tokens [B, gamma], fp32 uniforms
    [B, gamma+1], int32 outputs [B] and [B, gamma+1] and status [1]. NULL (None) operands are
    left to the library's own checks."""
    if not isinstance(target_logits, torch.Tensor) or target_logits.dim() != 3:
        raise ValueError("target_logits must be a [B, gamma+1, V] tensor")
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    if gamma < 0:
        raise ValueError("target_logits must have gamma+1 >= 1 positions")
    dtype_flag(target_logits)
    if draft_logits is not None:
        if draft_logits.dtype != target_logits.dtype:
            raise TypeError(f"draft_logits dtype {draft_logits.dtype} differs from "
                            f"target_logits dtype {target_logits.dtype}")
        _expect(draft_logits, "draft_logits", B * gamma * V, (target_logits.dtype,))
    _expect(draft_tokens, "draft_tokens", B * gamma, (torch.int32,))
    _expect(uniforms, "uniforms", B * (gamma + 1), (torch.float32,))
    _expect(accept_len, "accept_len", B, (torch.int32,))
    _expect(out_tokens, "out_tokens", B * (gamma + 1), (torch.int32,))
    _expect(status, "status", 1, (torch.int32,))
    return B, gamma, V


# ------------------------------------------------------------------ the C entry points

def spec_workspace_bytes(B: int, rows_per_b: int, V: int, dtype: int) -> int:
    return int(load_library().spec_workspace_bytes(B, rows_per_b, V, dtype))


def spec_workspace_init(workspace: torch.Tensor, stream=None) -> int:
    return load_library().spec_workspace_init(_ptr(workspace), _nbytes(workspace), _stream(stream))


def spec_verify_chain(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                      accept_len, out_tokens, status, workspace, stream=None) -> int:
    """target_logits [B, gamma+1, V], draft_logits [B, gamma, V] (fp32 or bf16), draft_tokens
    [B, gamma] int32, uniforms [B, gamma+1] fp32; outputs accept_len [B], out_tokens
    [B, gamma+1] int32; status [1] int32; workspace uint8 (scratch, no initialisation).
    Raises ValueError / TypeError when an operand's size or dtype does not match (B, gamma, V)."""
    B, gamma, V = _chain_shape_check(target_logits, draft_logits, draft_tokens, uniforms,
                                     temperature, accept_len, out_tokens, status)
    return load_library().spec_verify_chain(
        _ptr(target_logits), _ptr(draft_logits), dtype_flag(target_logits), _ptr(draft_tokens),
        _ptr(uniforms), B, gamma, V, float(temperature), _ptr(accept_len), _ptr(out_tokens),
        _ptr(status), _ptr(workspace), _nbytes(workspace), _stream(stream))


def spec_verify_chain_static(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                             accept_len, out_tokens, status, stream=None) -> int:
    """spec_verify_chain with the library's static scratch instead of a workspace (same
    operand checks)."""
    B, gamma, V = _chain_shape_check(target_logits, draft_logits, draft_tokens, uniforms,
                                     temperature, accept_len, out_tokens, status)
    return load_library().spec_verify_chain_static(
        _ptr(target_logits), _ptr(draft_logits), dtype_flag(target_logits), _ptr(draft_tokens),
        _ptr(uniforms), B, gamma, V, float(temperature), _ptr(accept_len), _ptr(out_tokens),
        _ptr(status), _stream(stream))


def spec_verify_tree(target_logits, parents, node_tokens, accept_len, path_nodes, out_tokens,
                     status, workspace, stream=None) -> int:
    """target_logits [B, N, V]; parents, node_tokens [B, N] int32; outputs accept_len [B],
    path_nodes [B, N], out_tokens [B, N] int32."""
    B, N, V = target_logits.shape
    return load_library().spec_verify_tree(
        _ptr(target_logits), dtype_flag(target_logits), _ptr(parents), _ptr(node_tokens), B, N,
        V, _ptr(accept_len), _ptr(path_nodes), _ptr(out_tokens), _ptr(status), _ptr(workspace),
        _nbytes(workspace), _stream(stream))


def spec_verify_tree_sample(target_logits, draft_logits, parents, node_tokens, uniforms,
                            temperature, accept_len, path_nodes, out_tokens, status, workspace,
                            stream=None) -> int:
    """target_logits, draft_logits [B, N, V]; parents, node_tokens [B, N] int32; uniforms [B, N]
    fp32 ([b, 0] the final draw, [b, i] node i's test); outputs as spec_verify_tree."""
    B, N, V = target_logits.shape
    if draft_logits is not None and (draft_logits.dtype != target_logits.dtype or
                                     tuple(draft_logits.shape) != (B, N, V)):
        raise ValueError("draft_logits must match target_logits in dtype and shape")
    _expect(uniforms, "uniforms", B * N, (torch.float32,))
    _expect(parents, "parents", B * N, (torch.int32,))
    _expect(node_tokens, "node_tokens", B * N, (torch.int32,))
    return load_library().spec_verify_tree_sample(
        _ptr(target_logits), _ptr(draft_logits), dtype_flag(target_logits), _ptr(parents),
        _ptr(node_tokens), _ptr(uniforms), B, N, V, float(temperature), _ptr(accept_len),
        _ptr(path_nodes), _ptr(out_tokens), _ptr(status), _ptr(workspace), _nbytes(workspace),
        _stream(stream))


def spec_lmhead_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return int(load_library().spec_lmhead_workspace_bytes(B, gamma, V))


def spec_verify_chain_lmhead(hidden_t, head_t, hidden_d, head_d, draft_tokens, uniforms,
                             temperature, logits_t, logits_d, accept_len, out_tokens, status,
                             workspace, stream=None) -> int:
    """hidden_t [B*(gamma+1), Ht], head_t [V, Ht], hidden_d [B*gamma, Hd], head_d [V, Hd] (bf16);
    draft_tokens [B, gamma] int32, uniforms [B, gamma+1] fp32; logits_t / logits_d bf16 outputs;
    accept_len [B], out_tokens [B, gamma+1] int32; status [1]; workspace uint8."""
    B, gamma = draft_tokens.shape
    V, Ht = head_t.shape
    Hd = head_d.shape[1]
    _expect(head_t, "head_t", V * Ht, (torch.bfloat16,))
    _expect(head_d, "head_d", V * Hd, (torch.bfloat16,))
    _expect(hidden_t, "hidden_t", B * (gamma + 1) * Ht, (torch.bfloat16,))
    _expect(hidden_d, "hidden_d", B * gamma * Hd, (torch.bfloat16,))
    _expect(logits_t, "logits_t", B * (gamma + 1) * V, (torch.bfloat16,))
    _expect(logits_d, "logits_d", B * gamma * V, (torch.bfloat16,))
    _expect(draft_tokens, "draft_tokens", B * gamma, (torch.int32,))
    _expect(uniforms, "uniforms", B * (gamma + 1), (torch.float32,))
    return load_library().spec_verify_chain_lmhead(
        _ptr(hidden_t), _ptr(head_t), Ht, _ptr(hidden_d), _ptr(head_d), Hd, _ptr(draft_tokens),
        _ptr(uniforms), B, gamma, V, float(temperature), _ptr(logits_t), _ptr(logits_d),
        _ptr(accept_len), _ptr(out_tokens), _ptr(status), _ptr(workspace), _nbytes(workspace),
        _stream(stream))


def spec_probs(logits, temperature, out_probs, status, workspace, stream=None) -> int:
    """logits [..., V] -> out_probs [..., V] fp32."""
    V = logits.shape[-1]
    rows = logits.numel() // V if V else 0
    return load_library().spec_probs(
        _ptr(logits), dtype_flag(logits), rows, V, float(temperature), _ptr(out_probs),
        _ptr(status), _ptr(workspace), _nbytes(workspace), _stream(stream))


def spec_launch_shape(kind: int, B: int, rows_per_b: int, V: int, dtype: int,
                      temperature: float = 1.0):
    """(kernels, grid, cluster) of a call of this shape on the current device."""
    k, g, c = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = load_library().spec_launch_shape(kind, B, rows_per_b, V, dtype, float(temperature),
                                          ctypes.byref(k), ctypes.byref(g), ctypes.byref(c))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_launch_shape")
    return k.value, g.value, c.value


def spec_sample(logits, temperature, uniforms, out_tokens, status, workspace, stream=None) -> int:
    """logits [rows, V] -> out_tokens [rows] int32 (uniforms [rows] fp32)."""
    V = logits.shape[-1]
    rows = logits.numel() // V if V else 0
    return load_library().spec_sample(
        _ptr(logits), dtype_flag(logits), rows, V, float(temperature), _ptr(uniforms),
        _ptr(out_tokens), _ptr(status), _ptr(workspace), _nbytes(workspace), _stream(stream))


def spec_topk(logits, k, out_idx, status, workspace, stream=None) -> int:
    """logits [rows, V] -> out_idx [rows, k] int32."""
    V = logits.shape[-1]
    rows = logits.numel() // V if V else 0
    return load_library().spec_topk(_ptr(logits), dtype_flag(logits), rows, V, int(k),
                                    _ptr(out_idx), _ptr(status), _ptr(workspace),
                                    _nbytes(workspace), _stream(stream))


def spec_tree_mask(parents, mask_words, status, stream=None) -> int:
    """parents [B, N] int32 -> mask_words [B, N, ceil(N/32)] (int32 tensor holding the bits)."""
    B, N = parents.shape
    return load_library().spec_tree_mask(_ptr(parents), B, N, _ptr(mask_words), _ptr(status),
                                         _stream(stream))


def spec_status_string(code: int) -> str:
    try:
        return load_library().spec_status_string(int(code)).decode()
    except ImportError:
        return f"status {code}"


def spec_last_cuda_error() -> int:
    """The cudaError_t behind this thread's last SPEC_ERR_LAUNCH (0 if none)."""
    try:
        return int(load_library().spec_last_cuda_error())
    except ImportError:
        return 0


def spec_cuda_error_string(cuda_error: int) -> str:
    return load_library().spec_cuda_error_string(int(cuda_error)).decode()


def spec_selftest_bounded_wait(status, limit_seconds: float, stream=None) -> int:
    """The bounded-wait self-check (see include/spec_verify.h): returns the SPEC_* code of the
    call; the kernel writes SPEC_ERR_TIMEOUT into status[0] when its waits give up."""
    _expect(status, "status", 1, (torch.int32,))
    return int(load_library().spec_selftest_bounded_wait(_ptr(status), float(limit_seconds),
                                                         _stream(stream)))


# ------------------------------------------------------------------ conveniences (allocation)

def new_workspace(B: int, rows_per_b: int, V: int, dtype: int, device=None) -> torch.Tensor:
    """A workspace tensor large enough for the given call shape (scratch; never needs zeroing)."""
    n = spec_workspace_bytes(B, rows_per_b, V, dtype)
    if n == 0:
        raise SpecError(SPEC_ERR_SHAPE, "spec_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def check(code: int, where: str) -> None:
    if code != SPEC_OK:
        raise SpecError(code, where)


def verify_chain(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                 workspace=None, stream=None):
    """Allocates the outputs and runs spec_verify_chain. Returns (accept_len, out_tokens,
    status) device tensors."""
    B, g1, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(B, 2 * (g1 - 1) + 1, V, dtype_flag(target_logits), dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, g1), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_verify_chain(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                            acc, out, st, workspace, stream), "spec_verify_chain")
    return acc, out, st


def verify_tree(target_logits, parents, node_tokens, workspace=None, stream=None):
    """Allocates the outputs and runs spec_verify_tree. Returns (accept_len, path_nodes,
    out_tokens, status) device tensors."""
    B, N, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(B, N, V, dtype_flag(target_logits), dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    out = torch.empty((B, N), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_verify_tree(target_logits, parents, node_tokens, acc, path, out, st, workspace,
                           stream), "spec_verify_tree")
    return acc, path, out, st


def verify_tree_sample(target_logits, draft_logits, parents, node_tokens, uniforms, temperature,
                       workspace=None, stream=None):
    """Allocates the outputs and runs spec_verify_tree_sample. Returns (accept_len, path_nodes,
    out_tokens, status) device tensors."""
    B, N, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = new_workspace(B, 2 * N, V, dtype_flag(target_logits), dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, N), dtype=torch.int32, device=dev)
    out = torch.empty((B, N), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_verify_tree_sample(target_logits, draft_logits, parents, node_tokens, uniforms,
                                  temperature, acc, path, out, st, workspace, stream),
          "spec_verify_tree_sample")
    return acc, path, out, st


def verify_chain_lmhead(hidden_t, head_t, hidden_d, head_d, draft_tokens, uniforms,
                        temperature, workspace=None, stream=None):
    """Allocates the outputs and runs spec_verify_chain_lmhead. Returns (accept_len, out_tokens,
    status, logits_t, logits_d) device tensors."""
    B, gamma = draft_tokens.shape
    V = head_t.shape[0]
    dev = hidden_t.device
    if workspace is None:
        n = spec_lmhead_workspace_bytes(B, gamma, V)
        if n == 0:
            raise SpecError(SPEC_ERR_SHAPE, "spec_lmhead_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    lt = torch.empty((B * (gamma + 1), V), dtype=torch.bfloat16, device=dev)
    ld = torch.empty((B * gamma, V), dtype=torch.bfloat16, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_verify_chain_lmhead(hidden_t, head_t, hidden_d, head_d, draft_tokens, uniforms,
                                   temperature, lt, ld, acc, out, st, workspace, stream),
          "spec_verify_chain_lmhead")
    return acc, out, st, lt, ld


def probs(logits, temperature, workspace=None, stream=None):
    """Allocates the output and runs spec_probs. Returns (probs fp32, status)."""
    V = logits.shape[-1]
    rows = logits.numel() // V
    dev = logits.device
    if workspace is None:
        workspace = new_workspace(rows, 1, V, dtype_flag(logits), dev)
    out = torch.empty(logits.shape, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_probs(logits, temperature, out, st, workspace, stream), "spec_probs")
    return out, st


def sample(logits, temperature, uniforms=None, workspace=None, stream=None):
    """Allocates the output and runs spec_sample. Returns (tokens [rows] int32, status)."""
    V = logits.shape[-1]
    rows = logits.numel() // V
    dev = logits.device
    if workspace is None:
        workspace = new_workspace(rows, 1, V, dtype_flag(logits), dev)
    out = torch.empty(rows, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_sample(logits, temperature, uniforms, out, st, workspace, stream), "spec_sample")
    return out, st


def topk(logits, k, workspace=None, stream=None):
    """Allocates the output and runs spec_topk. Returns (indices [rows, k] int32, status)."""
    V = logits.shape[-1]
    rows = logits.numel() // V
    dev = logits.device
    if workspace is None:
        workspace = new_workspace(rows, k, V, dtype_flag(logits), dev)
    out = torch.empty((rows, k), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    check(spec_topk(logits, k, out, st, workspace, stream), "spec_topk")
    return out, st


def tree_mask(parents, stream=None):
    """Allocates the output and runs spec_tree_mask. Returns (mask words [B, N, W] int32 holding
    the uint32 bit patterns, status)."""
    B, N = parents.shape
    W = (N + 31) // 32
    out = torch.empty((B, N, W), dtype=torch.int32, device=parents.device)
    st = torch.zeros(1, dtype=torch.int32, device=parents.device)
    check(spec_tree_mask(parents, out, st, stream), "spec_tree_mask")
    return out, st
