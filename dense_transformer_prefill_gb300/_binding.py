"""ctypes binding of include/dtp.h.  Argument marshalling only: torch tensors
supply device memory and the current CUDA stream; every computation happens in
libdtp.so's kernels."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB, build  # noqa: F401

DTP_F32, DTP_BF16, DTP_TF32 = 0, 1, 2
DTP_PREC_F32, DTP_PREC_TF32, DTP_PREC_BF16, DTP_PREC_E4M3 = 0, 1, 2, 3
KERNEL_KINDS = {"embed": 0, "rmsnorm": 1, "gemm_qkv": 2, "attn": 3, "gemm_o": 4,
                "gemm_gateup": 5, "gemm_down": 6, "gemm_lmhead": 7, "other": 8,
                "prompt": 9, "d2h": 10}

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


class DtpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dtp error {code}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("n_layer", c_int), ("n_embd", c_int), ("n_head", c_int), ("n_head_kv", c_int),
                ("head_dim", c_int), ("rope_dim_count", c_int), ("n_ff", c_int),
                ("n_vocab", c_int), ("rope_freq_base", c_float), ("rms_eps", c_float),
                ("precision", c_int), ("attn_gate", c_int)]


class LayerSrc(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                                       "ffn_norm", "w_gate", "w_up", "w_down")]


class FwdOutputs(ctypes.Structure):
    _fields_ = [("logits", c_void_p), ("last_only", c_int), ("hidden", c_void_p),
                ("k_cache", c_void_p), ("v_cache", c_void_p)]


_lib = None
_lock = threading.Lock()

_SIGS = {
    "dtp_last_error": ([], ctypes.c_char_p),
    "dtp_launch_count": ([c_int], ctypes.c_longlong),
    "dtp_packed_size": ([ctypes.POINTER(Config)], c_size_t),
    "dtp_pack_layer": ([ctypes.POINTER(Config), c_int, ctypes.POINTER(LayerSrc), c_void_p, c_size_t,
                        c_void_p], c_int),
    "dtp_pack_globals": ([ctypes.POINTER(Config), c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                          c_void_p], c_int),
    "dtp_workspace_size": ([ctypes.POINTER(Config), c_int], c_size_t),
    "dtp_workspace_size_host": ([ctypes.POINTER(Config), c_int], c_size_t),
    "dtp_fwd_prefill": ([ctypes.POINTER(Config), c_void_p, c_size_t, c_void_p, c_int, c_void_p,
                         c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "dtp_fwd_prefill_ex": ([ctypes.POINTER(Config), c_void_p, c_size_t, c_void_p, c_int,
                            ctypes.POINTER(FwdOutputs), c_void_p, c_size_t, c_void_p], c_int),
    "dtp_workspace_size_varlen": ([ctypes.POINTER(Config), c_int, c_int], c_size_t),
    "dtp_fwd_prefill_varlen": ([ctypes.POINTER(Config), c_void_p, c_size_t, c_void_p, c_void_p, c_int,
                                c_int, ctypes.POINTER(FwdOutputs), c_void_p, c_size_t, c_void_p],
                               c_int),
    "dtp_quantize_rows_e4m3": ([c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p], c_int),
    "dtp_rms_norm_e4m3": ([c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_float, c_void_p],
                          c_int),
    "dtp_linear_e4m3": ([c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int,
                         c_void_p, c_void_p], c_int),
    "dtp_workspace_size_host_batch": ([ctypes.POINTER(Config), c_int], c_size_t),
    "dtp_workspace_size_host_batch_n": ([ctypes.POINTER(Config), c_int, c_int], c_size_t),
    "dtp_fwd_prefill_host_batch": ([ctypes.POINTER(Config), c_void_p, c_size_t, c_void_p, c_int,
                                    c_int, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "dtp_kv_state_size": ([ctypes.POINTER(Config), c_int], c_size_t),
    "dtp_fwd_prefill_chunk": ([ctypes.POINTER(Config), c_void_p, c_size_t, c_void_p, c_int, c_int,
                               c_void_p, c_size_t, c_int, ctypes.POINTER(FwdOutputs), c_void_p,
                               c_size_t, c_void_p], c_int),
    "dtp_fwd_prefill_host": ([ctypes.POINTER(Config), c_void_p, c_size_t, c_void_p, c_int,
                              c_void_p, c_void_p, c_size_t, c_void_p], c_int),
    "dtp_check": ([c_void_p], c_int),
    "dtp_rms_norm": ([c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_float, c_void_p], c_int),
    "dtp_qk_norm_rope_neox": ([c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                               c_float, c_float, c_void_p], c_int),
    "dtp_sdpa_workspace_size": ([c_int, c_int, c_int, c_int], c_size_t),
    "dtp_sdpa_causal_gqa": ([c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                             c_int, c_float, c_void_p, c_size_t, c_void_p], c_int),
    "dtp_swiglu": ([c_void_p, c_void_p, c_void_p, c_int, c_size_t, c_void_p], c_int),
    "dtp_linear": ([c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p,
                    c_void_p], c_int),
    "dtp_qkv_norm_rope_workspace_size": ([c_int, c_int], c_size_t),
    "dtp_qkv_norm_rope": ([c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                           c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_float,
                           c_void_p, c_size_t, c_void_p], c_int),
    "dtp_gate_up_swiglu": ([c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_void_p], c_int),
    "dtp_selftest_wait_timeout": ([c_void_p], c_int),
    "dtp_timer_enable": ([ctypes.c_uint, c_int], c_int),
    "dtp_timer_disable": ([], c_int),
    "dtp_timer_read": ([c_int, ctypes.POINTER(c_int), ctypes.POINTER(c_float)], c_int),
    "dtp_timer_spans": ([c_int, c_int, c_int, ctypes.POINTER(c_float), ctypes.POINTER(c_float),
                         ctypes.POINTER(c_int)], c_int),
}


def lib():
    """The loaded libdtp.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"{LIB} is not built; call dense_transformer_prefill_gb300.build()")
            L = ctypes.CDLL(LIB)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def last_error() -> str:
    return lib().dtp_last_error().decode()


def _ok(rc: int) -> None:
    if rc != 0:
        raise DtpError(rc, last_error())


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTP_F32
    if t.dtype == torch.bfloat16:
        return DTP_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def config_from(cfg) -> Config:
    """Config from an object/dict with the dtp_config field names; precision may be
    "f32"/"tf32"/"bf16"/"e4m3" or the DTP_PREC_* code."""
    get = (lambda k: cfg[k]) if isinstance(cfg, dict) else (lambda k: getattr(cfg, k))
    prec = get("precision")
    if isinstance(prec, str):
        prec = {"f32": DTP_PREC_F32, "tf32": DTP_PREC_TF32, "bf16": DTP_PREC_BF16,
                "e4m3": DTP_PREC_E4M3}[prec]
    try:
        gate = int(bool(get("attn_gate")))
    except (KeyError, AttributeError):
        gate = 0
    return Config(get("n_layer"), get("n_embd"), get("n_head"), get("n_head_kv"), get("head_dim"),
                  get("rope_dim_count"), get("n_ff"), get("n_vocab"), float(get("rope_freq_base")),
                  float(get("rms_eps")), prec, gate)


# ----------------------------------------------------------------------------- entry points
def packed_size(c: Config) -> int:
    return lib().dtp_packed_size(ctypes.byref(c))


def workspace_size(c: Config, T: int) -> int:
    return lib().dtp_workspace_size(ctypes.byref(c), T)


def workspace_size_host(c: Config, T: int) -> int:
    return lib().dtp_workspace_size_host(ctypes.byref(c), T)


def pack_layer(c: Config, layer: int, src: dict, packed: torch.Tensor, stream=None) -> None:
    s = LayerSrc(*[_ptr(src[n]) for n, _ in LayerSrc._fields_])
    _ok(lib().dtp_pack_layer(ctypes.byref(c), layer, ctypes.byref(s), packed.data_ptr(),
                             packed.numel() * packed.element_size(), _stream(stream)))


def pack_globals(c: Config, tok_embd, output_norm, output, packed: torch.Tensor, stream=None) -> None:
    _ok(lib().dtp_pack_globals(ctypes.byref(c), _ptr(tok_embd), _ptr(output_norm), _ptr(output),
                               packed.data_ptr(), packed.numel() * packed.element_size(),
                               _stream(stream)))


def fwd_prefill(c: Config, packed: torch.Tensor, tokens: torch.Tensor, logits: torch.Tensor,
                workspace: torch.Tensor, hidden: torch.Tensor | None = None, stream=None) -> None:
    assert tokens.dtype in (torch.int32, torch.uint32) and tokens.is_contiguous()
    assert logits.dtype == torch.float32 and logits.is_contiguous()
    _ok(lib().dtp_fwd_prefill(ctypes.byref(c), packed.data_ptr(),
                              packed.numel() * packed.element_size(), tokens.data_ptr(),
                              tokens.numel(), logits.data_ptr(), _ptr(hidden),
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream(stream)))


def fwd_prefill_ex(c: Config, packed: torch.Tensor, tokens: torch.Tensor, workspace: torch.Tensor,
                   logits=None, last_only: bool = False, hidden=None, k_cache=None, v_cache=None,
                   stream=None) -> None:
    o = FwdOutputs(_ptr(logits), 1 if last_only else 0, _ptr(hidden), _ptr(k_cache), _ptr(v_cache))
    _ok(lib().dtp_fwd_prefill_ex(ctypes.byref(c), packed.data_ptr(),
                                 packed.numel() * packed.element_size(), tokens.data_ptr(),
                                 tokens.numel(), ctypes.byref(o), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def workspace_size_varlen(c: Config, total: int, n_seq: int) -> int:
    return lib().dtp_workspace_size_varlen(ctypes.byref(c), total, n_seq)


def fwd_prefill_varlen(c: Config, packed: torch.Tensor, tokens: torch.Tensor,
                       cu_seqlens: torch.Tensor, workspace: torch.Tensor, logits=None,
                       last_only: bool = False, hidden=None, k_cache=None, v_cache=None,
                       stream=None) -> None:
    assert cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous()
    o = FwdOutputs(_ptr(logits), 1 if last_only else 0, _ptr(hidden), _ptr(k_cache), _ptr(v_cache))
    _ok(lib().dtp_fwd_prefill_varlen(ctypes.byref(c), packed.data_ptr(),
                                     packed.numel() * packed.element_size(), tokens.data_ptr(),
                                     cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, tokens.numel(),
                                     ctypes.byref(o), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def kv_state_size(c: Config, max_T: int) -> int:
    return lib().dtp_kv_state_size(ctypes.byref(c), max_T)


def fwd_prefill_chunk(c: Config, packed: torch.Tensor, tokens: torch.Tensor, p0: int,
                      kv_state: torch.Tensor, max_T: int, workspace: torch.Tensor, logits=None,
                      last_only: bool = False, hidden=None, stream=None) -> None:
    """Positions p0 .. p0+len(tokens)-1 of one sequence against `kv_state`
    (dtp_kv_state_size(c, max_T) bytes), which holds positions 0 .. p0-1."""
    assert tokens.dtype in (torch.int32, torch.uint32) and tokens.is_contiguous()
    o = FwdOutputs(_ptr(logits), 1 if last_only else 0, _ptr(hidden), None, None)
    _ok(lib().dtp_fwd_prefill_chunk(ctypes.byref(c), packed.data_ptr(),
                                    packed.numel() * packed.element_size(), tokens.data_ptr(),
                                    tokens.numel(), p0, kv_state.data_ptr(),
                                    kv_state.numel() * kv_state.element_size(), max_T,
                                    ctypes.byref(o), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream)))


def fwd_prefill_host(c: Config, packed: torch.Tensor, tokens_host: torch.Tensor,
                     logits_host: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    assert tokens_host.device.type == "cpu" and logits_host.device.type == "cpu"
    _ok(lib().dtp_fwd_prefill_host(ctypes.byref(c), packed.data_ptr(),
                                   packed.numel() * packed.element_size(), tokens_host.data_ptr(),
                                   tokens_host.numel(), logits_host.data_ptr(),
                                   workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))


def workspace_size_host_batch(c: Config, T: int, n_buffers: int = 2) -> int:
    """Workspace bytes for fwd_prefill_host_batch with n_buffers (2..8) device
    logit buffers; 0 when n_buffers is out of range."""
    if n_buffers == 2:
        return lib().dtp_workspace_size_host_batch(ctypes.byref(c), T)
    return lib().dtp_workspace_size_host_batch_n(ctypes.byref(c), T, n_buffers)


def fwd_prefill_host_batch(c: Config, packed: torch.Tensor, tokens_host: list, logits_host: list,
                           workspace: torch.Tensor, stream=None) -> None:
    """n prompts host to host; the logits copy of prompt j overlaps the forward
    pass of prompt j + 1.  tokens_host: n CPU uint32/int32 tensors [T];
    logits_host: n CPU float32 tensors [T, n_vocab] (pinned for asynchronous copies)."""
    n = len(tokens_host)
    assert n == len(logits_host) and n > 0
    T = tokens_host[0].numel()
    for t, lg in zip(tokens_host, logits_host):
        assert t.device.type == "cpu" and t.numel() == T and t.is_contiguous()
        assert lg.device.type == "cpu" and lg.dtype == torch.float32 and lg.is_contiguous()
    toks = (c_void_p * n)(*[t.data_ptr() for t in tokens_host])
    logs = (c_void_p * n)(*[lg.data_ptr() for lg in logits_host])
    _ok(lib().dtp_fwd_prefill_host_batch(ctypes.byref(c), packed.data_ptr(),
                                         packed.numel() * packed.element_size(), toks, n, T, logs,
                                         workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def check(stream=None) -> None:
    _ok(lib().dtp_check(_stream(stream)))


def rms_norm(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, eps: float, tf32: bool = False,
             stream=None) -> None:
    """tf32=True: float32 y rounded to tf32 (a tensor-core GEMM operand)."""
    rows, cols = x.shape
    dt = DTP_TF32 if tf32 else _dtype_code(y)
    _ok(lib().dtp_rms_norm(x.data_ptr(), w.data_ptr(), y.data_ptr(), dt, rows, cols,
                           eps, _stream(stream)))


def qk_norm_rope_neox(x: torch.Tensor, w_norm, pos, n_heads: int, head_dim: int,
                      rope_dim_count: int, freq_base: float, eps: float, stream=None) -> None:
    _ok(lib().dtp_qk_norm_rope_neox(x.data_ptr(), _dtype_code(x), _ptr(w_norm), _ptr(pos),
                                    x.shape[0], n_heads, head_dim, rope_dim_count, freq_base, eps,
                                    _stream(stream)))


def sdpa_workspace_size(T: int, n_head_kv: int, head_dim: int, dtype: int) -> int:
    return lib().dtp_sdpa_workspace_size(T, n_head_kv, head_dim, dtype)


def sdpa_causal_gqa(q, k, v, out, n_head: int, n_head_kv: int, head_dim: int, scale: float,
                    workspace=None, tf32: bool = False, stream=None) -> None:
    """tf32=True: float32 q/k/v holding tf32 values on the tcgen05 kind::tf32 kernel."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    dt = DTP_TF32 if tf32 else _dtype_code(q)
    _ok(lib().dtp_sdpa_causal_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  dt, q.shape[0], n_head, n_head_kv, head_dim, scale,
                                  _ptr(workspace), ws_bytes, _stream(stream)))


def swiglu(gate, up, out, stream=None) -> None:
    _ok(lib().dtp_swiglu(gate.data_ptr(), up.data_ptr(), out.data_ptr(), _dtype_code(gate),
                         gate.numel(), _stream(stream)))


def linear(x, W, y, residual=None, tf32: bool = False, stream=None) -> None:
    """y = x W^T (+ residual).  tf32=True: float32 x and W holding tf32 values
    go to the kind::tf32 tensor-core GEMM."""
    M, K = x.shape
    N = W.shape[0]
    dt = DTP_TF32 if tf32 else _dtype_code(x)
    _ok(lib().dtp_linear(x.data_ptr(), W.data_ptr(), y.data_ptr(), dt, _dtype_code(y),
                         M, N, K, _ptr(residual), _stream(stream)))


def quantize_rows_e4m3(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, stream=None) -> None:
    """Per-row e4m3 codes (uint8 [rows, cols]) and float32 scales [rows] of x."""
    rows, cols = x.shape
    _ok(lib().dtp_quantize_rows_e4m3(x.data_ptr(), _dtype_code(x), rows, cols, q.data_ptr(),
                                     scale.data_ptr(), _stream(stream)))


def rms_norm_e4m3(x: torch.Tensor, w: torch.Tensor, q: torch.Tensor, scale: torch.Tensor,
                  eps: float, stream=None) -> None:
    rows, cols = x.shape
    _ok(lib().dtp_rms_norm_e4m3(x.data_ptr(), w.data_ptr(), q.data_ptr(), scale.data_ptr(), rows,
                                cols, eps, _stream(stream)))


def linear_e4m3(xq, x_scale, wq, w_scale, y, residual=None, stream=None) -> None:
    """y = x_scale[m] w_scale[n] (xq wq^T)[m, n] (+ residual) on e4m3 codes."""
    M, K = xq.shape
    N = wq.shape[0]
    _ok(lib().dtp_linear_e4m3(xq.data_ptr(), x_scale.data_ptr(), wq.data_ptr(), w_scale.data_ptr(),
                              y.data_ptr(), M, N, K, _ptr(residual), _stream(stream)))


def qkv_norm_rope(h, w_qkv, q_norm, k_norm, q, k, vt, n_head: int, n_head_kv: int,
                  head_dim: int, rope_dim_count: int, freq_base: float, eps: float,
                  workspace=None, stream=None) -> None:
    T, d = h.shape
    if workspace is None:
        workspace = torch.empty(lib().dtp_qkv_norm_rope_workspace_size(T, rope_dim_count),
                                dtype=torch.uint8, device=h.device)
    _ok(lib().dtp_qkv_norm_rope(h.data_ptr(), w_qkv.data_ptr(), q_norm.data_ptr(), k_norm.data_ptr(),
                                q.data_ptr(), k.data_ptr(), vt.data_ptr(), vt.shape[1], T, d, n_head,
                                n_head_kv, head_dim, rope_dim_count, freq_base, eps,
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream(stream)))


def gate_up_swiglu(z, w_gu, act, stream=None) -> None:
    T, d = z.shape
    _ok(lib().dtp_gate_up_swiglu(z.data_ptr(), w_gu.data_ptr(), act.data_ptr(), T, d, act.shape[1],
                                 _stream(stream)))


def selftest_wait_timeout(stream=None) -> None:
    _ok(lib().dtp_selftest_wait_timeout(_stream(stream)))


def timer_enable(kinds, capacity: int) -> None:
    mask = 0
    for k in kinds:
        mask |= 1 << (KERNEL_KINDS[k] if isinstance(k, str) else k)
    _ok(lib().dtp_timer_enable(mask, capacity))


def timer_disable() -> None:
    _ok(lib().dtp_timer_disable())


def timer_read(kind) -> tuple[int, float]:
    n, ms = c_int(0), c_float(0.0)
    _ok(lib().dtp_timer_read(KERNEL_KINDS[kind] if isinstance(kind, str) else kind,
                             ctypes.byref(n), ctypes.byref(ms)))
    return n.value, ms.value


def timer_spans(kind, ref_kind, cap: int = 4096) -> list[tuple[float, float]]:
    """(start, end) in ms of each recorded launch or span of `kind`, measured from
    the start of the first recorded one of `ref_kind`."""
    k = KERNEL_KINDS[kind] if isinstance(kind, str) else kind
    r = KERNEL_KINDS[ref_kind] if isinstance(ref_kind, str) else ref_kind
    st, en, n = (c_float * cap)(), (c_float * cap)(), c_int(0)
    _ok(lib().dtp_timer_spans(k, r, cap, st, en, ctypes.byref(n)))
    return [(st[i], en[i]) for i in range(min(n.value, cap))]


def launch_count(reset: bool = False) -> int:
    return lib().dtp_launch_count(1 if reset else 0)


# ----------------------------------------------------------------------------- model holder
class Model:
    """Owns the packed weight buffer (and cached workspaces) of one model on one device."""

    def __init__(self, cfg, device="cuda"):
        self.cfg = cfg
        self.c = config_from(cfg)
        self.device = torch.device(device)
        n = packed_size(self.c)
        if n == 0:
            raise DtpError(-1, last_error())
        self.packed = torch.empty(n, dtype=torch.uint8, device=self.device)
        self._ws = {}

    def load_layer(self, layer: int, arrays: dict, stream=None) -> None:
        """Pack one layer from float32 arrays (numpy or torch) with the dtp_layer_src names."""
        dev = {k: torch.as_tensor(v).to(self.device, torch.float32).contiguous()
               for k, v in arrays.items()}
        pack_layer(self.c, layer, dev, self.packed, stream)
        torch.cuda.current_stream(self.device).synchronize()

    def load_globals(self, tok_embd, output_norm, output, stream=None) -> None:
        t = [torch.as_tensor(a).to(self.device, torch.float32).contiguous()
             for a in (tok_embd, output_norm, output)]
        pack_globals(self.c, *t, self.packed, stream)
        torch.cuda.current_stream(self.device).synchronize()

    def workspace(self, T: int, host: bool = False) -> torch.Tensor:
        key = (T, host)
        if key not in self._ws:
            n = (workspace_size_host if host else workspace_size)(self.c, T)
            if n == 0:
                raise DtpError(-1, last_error())
            self._ws[key] = torch.empty(n, dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def workspace_varlen(self, total: int, n_seq: int) -> torch.Tensor:
        key = ("varlen", total, n_seq)
        if key not in self._ws:
            n = workspace_size_varlen(self.c, total, n_seq)
            if n == 0:
                raise DtpError(-1, last_error())
            self._ws[key] = torch.empty(n, dtype=torch.uint8, device=self.device)
        return self._ws[key]

    def forward(self, tokens: torch.Tensor, logits: torch.Tensor | None = None,
                hidden: bool | torch.Tensor = False, stream=None):
        T = tokens.numel()
        if logits is None:
            logits = torch.empty((T, self.c.n_vocab), dtype=torch.float32, device=self.device)
        hid = None
        if hidden is True:
            hid = torch.empty((self.c.n_layer + 1, T, self.c.n_embd), dtype=torch.float32,
                              device=self.device)
        elif isinstance(hidden, torch.Tensor):
            hid = hidden
        fwd_prefill(self.c, self.packed, tokens, logits, self.workspace(T), hid, stream)
        return (logits, hid) if hid is not None else logits
