"""ctypes binding of libescha.so, the C ABI declared in include/escha.h.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI. Torch tensors provide device memory and the current
stream. There is no CPU fallback: if the library is missing or the device is
not an sm_103 GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libescha.so")

ESCHA_OK = 0
ESCHA_E_ARG = -1
ESCHA_E_SHAPE = -2
ESCHA_E_K = -3
ESCHA_E_WORKSPACE = -4
ESCHA_E_ALIGN = -5
ESCHA_E_CUDA = -6
ESCHA_E_DEVICE = -7
ESCHA_E_CKPT = -8
ESCHA_E_IO = -9

ESCHA_PATH_FUSED = 1
ESCHA_PATH_SLOT = 2
ESCHA_PATH_GROUPED = 3
ESCHA_PATH_SEQUENCE = 4

ESCHA_F16 = 1
ESCHA_BF16 = 2
ESCHA_F32 = 3

EXPORTS = [
    "escha_last_error",
    "escha_version",
    "escha_trellis_decode",
    "escha_trellis_gemv_workspace",
    "escha_trellis_gemv",
    "escha_codes_to_nt_major",
    "escha_dense_linear_workspace",
    "escha_dense_linear",
    "escha_ckpt_open",
    "escha_ckpt_close",
    "escha_ckpt_num_projections",
    "escha_ckpt_projection",
    "escha_ckpt_tensor_info",
    "escha_ckpt_read",
    "escha_ckpt_load_projection",
    "escha_moe_block_workspace",
    "escha_moe_block",
    "escha_moe_block_timed",
    "escha_moe_block_resid",
    "escha_moe_block_noalloc",
    "escha_moe_seq_workspace",
    "escha_moe_blocks",
    "escha_moe_stack",
    "escha_moe_block_path",
    "escha_moe_blocks_path",
    "escha_moe_blocks_timed",
    "escha_debug_set_blocks_route",
    "escha_debug_set_moe_route",
    "escha_debug_set_fused_wait",
    "escha_debug_set_cluster_wait",
    "escha_moe_route_workspace",
    "escha_moe_route",
    "escha_residual_rmsnorm",
    "int8_w8a16_workspace",
    "int8_w8a16_matvec",
    "int8_w8a16_dequant",
]

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t


class EschaMoeLayer(ctypes.Structure):
    """Mirror of ``escha_moe_layer`` in include/escha.h."""

    _fields_ = [
        ("hidden", _i),
        ("inter", _i),
        ("n_experts", _i),
        ("topk", _i),
        ("router_w", _vp),
        ("gu_codes", _vp),
        ("gu_K", _i),
        ("gu_rin", _vp),
        ("gu_rout", _vp),
        ("dn_codes", _vp),
        ("dn_K", _i),
        ("dn_rin", _vp),
        ("dn_rout", _vp),
        ("sh_inter", _i),
        ("sh_gu_w8", _vp),
        ("sh_gu_scale", _vp),
        ("sh_dn_w8", _vp),
        ("sh_dn_scale", _vp),
        ("sh_gate", _vp),
    ]


class EschaProjInfo(ctypes.Structure):
    """Mirror of ``escha_proj_info`` in include/escha.h."""

    _fields_ = [
        ("prefix", ctypes.c_char * 256),
        ("K", _i),
        ("n_experts", _i),
        ("n_in", _i),
        ("n_out", _i),
        ("has_bias", _i),
        ("has_s_in", _i),
        ("has_s_out", _i),
        ("has_config", _i),
        ("scales_all_ones", _i),
        ("config_k", _i),
    ]


class EschaTensorInfo(ctypes.Structure):
    """Mirror of ``escha_tensor_info`` in include/escha.h."""

    _fields_ = [("dtype", ctypes.c_char * 8), ("ndim", _i), ("shape", ctypes.c_longlong * 8), ("nbytes", _sz)]


_LIB = None


def lib() -> ctypes.CDLL:
    """Load libescha.so once (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(python -m bit_trellis_quantized_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        L.escha_last_error.restype = ctypes.c_char_p
        L.escha_last_error.argtypes = []
        L.escha_version.restype = _i
        L.escha_trellis_decode.argtypes = [_vp, _i, _i, _i, _vp, _vp]
        L.escha_trellis_decode.restype = _i
        L.escha_trellis_gemv_workspace.argtypes = [_i, _i, _i, _i]
        L.escha_trellis_gemv_workspace.restype = _sz
        L.escha_trellis_gemv.argtypes = [_vp, _i, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]
        L.escha_trellis_gemv.restype = _i
        L.escha_codes_to_nt_major.argtypes = [_vp, _i, _i, _i, _vp, _vp]
        L.escha_codes_to_nt_major.restype = _i
        L.escha_dense_linear_workspace.argtypes = [_i, _i, _i, _i]
        L.escha_dense_linear_workspace.restype = _sz
        L.escha_dense_linear.argtypes = [_vp, _i, _i, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.escha_dense_linear.restype = _i
        L.escha_ckpt_open.argtypes = [ctypes.POINTER(ctypes.c_char_p), _i, ctypes.POINTER(_vp)]
        L.escha_ckpt_open.restype = _i
        L.escha_ckpt_close.argtypes = [_vp]
        L.escha_ckpt_close.restype = None
        L.escha_ckpt_num_projections.argtypes = [_vp]
        L.escha_ckpt_num_projections.restype = _i
        L.escha_ckpt_projection.argtypes = [_vp, _i, ctypes.POINTER(EschaProjInfo)]
        L.escha_ckpt_projection.restype = _i
        L.escha_ckpt_tensor_info.argtypes = [_vp, ctypes.c_char_p, ctypes.POINTER(EschaTensorInfo)]
        L.escha_ckpt_tensor_info.restype = _i
        L.escha_ckpt_read.argtypes = [_vp, ctypes.c_char_p, _vp, _sz, _i, _vp]
        L.escha_ckpt_read.restype = _i
        L.escha_ckpt_load_projection.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _i, _vp]
        L.escha_ckpt_load_projection.restype = _i
        L.escha_moe_block_workspace.argtypes = [ctypes.POINTER(EschaMoeLayer), _i]
        L.escha_moe_block_workspace.restype = _sz
        L.escha_moe_block.argtypes = [ctypes.POINTER(EschaMoeLayer), _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp]
        L.escha_moe_block.restype = _i
        L.escha_moe_block_timed.argtypes = [ctypes.POINTER(EschaMoeLayer), _vp, _i, _vp, _vp, _vp, _vp, _sz, _vp,
                                            ctypes.POINTER(_vp)]
        L.escha_moe_block_timed.restype = _i
        L.escha_moe_block_resid.argtypes = [ctypes.POINTER(EschaMoeLayer), _vp, _vp, ctypes.c_float, _vp, _i, _vp, _vp,
                                            _vp, _vp, _sz, _vp]
        L.escha_moe_block_resid.restype = _i
        L.escha_moe_block_noalloc.argtypes = [ctypes.POINTER(EschaMoeLayer), _vp, _i, _vp, _vp, _vp, _vp]
        L.escha_moe_block_noalloc.restype = _i
        _lp = ctypes.POINTER(ctypes.POINTER(EschaMoeLayer))
        L.escha_moe_seq_workspace.argtypes = [_lp, _i]
        L.escha_moe_seq_workspace.restype = _sz
        L.escha_moe_blocks.argtypes = [_lp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                       ctypes.POINTER(_vp), _vp, _sz, _vp]
        L.escha_moe_blocks.restype = _i
        L.escha_moe_stack.argtypes = [_lp, _i, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
        L.escha_moe_stack.restype = _i
        L.escha_moe_block_path.argtypes = [ctypes.POINTER(EschaMoeLayer), _i]
        L.escha_moe_block_path.restype = _i
        L.escha_moe_blocks_timed.argtypes = [_lp, _i, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                             ctypes.POINTER(_vp), _vp, _sz, _vp, ctypes.POINTER(_vp)]
        L.escha_moe_blocks_timed.restype = _i
        L.escha_moe_blocks_path.argtypes = [_lp, _i]
        L.escha_moe_blocks_path.restype = _i
        L.escha_debug_set_blocks_route.argtypes = [_i]
        L.escha_debug_set_blocks_route.restype = _i
        L.escha_debug_set_moe_route.argtypes = [_i]
        L.escha_debug_set_moe_route.restype = _i
        L.escha_debug_set_fused_wait.argtypes = [ctypes.c_longlong, _i]
        L.escha_debug_set_fused_wait.restype = _i
        L.escha_debug_set_cluster_wait.argtypes = [_i, _i]
        L.escha_debug_set_cluster_wait.restype = _i
        L.escha_moe_route_workspace.argtypes = [ctypes.POINTER(EschaMoeLayer), _i]
        L.escha_moe_route_workspace.restype = _sz
        L.escha_moe_route.argtypes = [ctypes.POINTER(EschaMoeLayer), _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                      _vp]
        L.escha_moe_route.restype = _i
        L.escha_residual_rmsnorm.argtypes = [_vp, _vp, _i, _i, ctypes.c_float, _vp, _vp]
        L.escha_residual_rmsnorm.restype = _i
        L.int8_w8a16_workspace.argtypes = [_i, _i, _i]
        L.int8_w8a16_workspace.restype = _sz
        L.int8_w8a16_matvec.argtypes = [_vp, _vp, _i, _i, _vp, _i, _i, _vp, _vp, _sz, _vp]
        L.int8_w8a16_matvec.restype = _i
        L.int8_w8a16_dequant.argtypes = [_vp, _vp, _i, _i, _vp, _vp]
        L.int8_w8a16_dequant.restype = _i
        _LIB = L
    return _LIB


def set_moe_route(mode: int) -> None:
    """Diagnostic: 0 = one-token blocks run the fused single kernel where it
    applies, 1 = always the three per-slot kernels, 2 = always the fused one."""
    check(lib().escha_debug_set_moe_route(int(mode)))


def set_blocks_route(mode: int = 0) -> None:
    """Diagnostic: escha_moe_blocks by shape (0), forced onto the per-slot
    kernels over all blocks (1) or onto the sequence kernel (2)."""
    check(lib().escha_debug_set_blocks_route(int(mode)))


def set_fused_wait(wait_ns: int = 2_000_000_000, skip_publish: bool = False) -> None:
    """Diagnostic: the fused kernel's wait bound, and the test hook that keeps
    the routing unpublished so that every wait on it runs out."""
    check(lib().escha_debug_set_fused_wait(int(wait_ns), int(bool(skip_publish))))


def set_cluster_wait(poll_limit_log2: int = 24, skip_arrive: bool = False) -> None:
    """Diagnostic: the per-slot cluster reductions' wait bound (2^poll_limit_log2
    polls), and the test hook that keeps ranks != 0 from storing or arriving
    so that rank 0's wait runs out."""
    check(lib().escha_debug_set_cluster_wait(int(poll_limit_log2), int(bool(skip_arrive))))


class EschaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"escha error {code}: {msg}")
        self.code = code


def check(code: int) -> None:
    if code != ESCHA_OK:
        raise EschaError(code, lib().escha_last_error().decode())


def ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_tag(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return ESCHA_F16
    if t.dtype == torch.bfloat16:
        return ESCHA_BF16
    if t.dtype == torch.float32:
        return ESCHA_F32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# --------------------------------------------------------------------------
# High-level wrappers (torch tensors in, torch tensors out).
# --------------------------------------------------------------------------


def trellis_decode(codes: torch.Tensor, stream=None) -> torch.Tensor:
    """Dense fp16 weights W[in][out] of a code tensor [in/16][out/16][16K]."""
    _need_cuda(codes)
    KT, NT, L = codes.shape
    W = torch.empty((KT * 16, NT * 16), dtype=torch.float16, device=codes.device)
    check(lib().escha_trellis_decode(ptr(codes), KT * 16, NT * 16, L // 16, ptr(W), stream_handle(stream)))
    return W


def trellis_gemv(codes, x, rin, rout, y=None, stream=None) -> torch.Tensor:
    """y[b] = rout * H(W^T H(rin * x[b])) for a batch of tokens sharing one
    trellis-coded weight. x: [batch][in] fp16 or f32."""
    _need_cuda(codes, x, rin, rout)
    KT, NT, L = codes.shape
    n_in, n_out = KT * 16, NT * 16
    if x.dim() == 1:
        x = x.unsqueeze(0)
    batch = x.shape[0]
    if y is None:
        y = torch.empty((batch, n_out), dtype=torch.float32, device=x.device)
    check(lib().escha_trellis_gemv(ptr(codes), n_in, n_out, L // 16, ptr(x), _dtype_tag(x), batch, ptr(rin),
                                   ptr(rout), ptr(y), None, 0, stream_handle(stream)))
    return y


def codes_to_nt_major(codes: torch.Tensor, stream=None) -> torch.Tensor:
    """Whole-tile transpose of a code tensor [in/16][out/16][16K] to the
    nt-major grid [out/16][in/16][16K] (a load-time step)."""
    _need_cuda(codes)
    KT, NT, L = codes.shape
    dst = torch.empty((NT, KT, L), dtype=codes.dtype, device=codes.device)
    check(lib().escha_codes_to_nt_major(ptr(codes), KT * 16, NT * 16, L // 16, ptr(dst), stream_handle(stream)))
    return dst


class DenseLinear:
    """One trellis-coded dense projection y = rout * H(W^T H(rin * x)) + bias.

    ``codes`` is the stored kt-major tensor [in/16][out/16][16K]; with
    ``nt_major=True`` it is transposed once here and the kernels walk the
    nt-major grid. ``bias`` (f32 [out]) is optional."""

    def __init__(self, codes, rin, rout, bias=None, nt_major: bool = True, stream=None):
        _need_cuda(codes, rin, rout)
        KT, NT, L = codes.shape
        self.n_in, self.n_out, self.K = KT * 16, NT * 16, L // 16
        self.nt_major = bool(nt_major)
        self.codes = codes_to_nt_major(codes, stream) if self.nt_major else codes
        if self.nt_major:
            # the transposed codes are weights, which the kernels read before
            # their programmatic-launch wait: finish the load-time copy first
            (stream if stream is not None else torch.cuda.current_stream(codes.device)).synchronize()
        self.rin, self.rout = rin, rout
        self.bias = bias.contiguous() if bias is not None else None
        self._ws = None

    @classmethod
    def from_checkpoint(cls, ckpt: "Checkpoint", i: int, device="cuda", nt_major: bool = True, stream=None):
        """Dense projection i of an opened checkpoint, its tiles moved to the
        nt-major grid at load (nt_major) and its bias, if any, widened to f32."""
        ld = ckpt.load_projection(i, device=device, nt_major=nt_major, stream=stream)
        p = ld["info"]
        if p["n_experts"]:
            raise ValueError(f"{p['prefix']} holds stacked experts, not a dense projection")
        self = cls.__new__(cls)
        self.n_in, self.n_out, self.K, self.nt_major = p["in"], p["out"], p["K"], bool(nt_major)
        self.codes, self.rin, self.rout, self.bias = ld["codes"], ld["rin"], ld["rout"], ld["bias"]
        self._ws = None
        return self

    def workspace_bytes(self, M: int) -> int:
        return lib().escha_dense_linear_workspace(self.n_in, self.n_out, self.K, M)

    def __call__(self, x, y=None, ws=None, stream=None) -> torch.Tensor:
        if x.dim() == 1:
            x = x.unsqueeze(0)
        _need_cuda(x)
        M = x.shape[0]
        if y is None:
            y = torch.empty((M, self.n_out), dtype=torch.float32, device=x.device)
        nbytes = self.workspace_bytes(M)
        if ws is None:
            if self._ws is None or self._ws.numel() < nbytes:
                self._ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
            ws = self._ws
        check(lib().escha_dense_linear(ptr(self.codes), self.n_in, self.n_out, self.K, int(self.nt_major), ptr(x),
                                       _dtype_tag(x), M, ptr(self.rin), ptr(self.rout),
                                       ptr(self.bias) if self.bias is not None else None, ptr(y), ptr(ws),
                                       ws.numel(), stream_handle(stream)))
        return y

    def status(self) -> int:
        """The status word of the last call (0: every bounded wait completed)."""
        return int(self._ws[:4].view(torch.int32).item()) if self._ws is not None else 0


_ST_DTYPES = {"F16": np.float16, "BF16": np.uint16, "F32": np.float32, "F64": np.float64, "I8": np.int8,
              "U8": np.uint8, "I16": np.int16, "U16": np.uint16, "I32": np.int32, "U32": np.uint32,
              "I64": np.int64, "U64": np.uint64, "BOOL": np.bool_}


class Checkpoint:
    """Safetensors shards of an Escha-W2 export, opened through the native
    loader, which checks the escha leaf contract on open (EschaError with
    code ESCHA_E_CKPT / ESCHA_E_IO otherwise)."""

    def __init__(self, paths):
        if isinstance(paths, (str, os.PathLike)):
            paths = [paths]
        enc = [os.fspath(p).encode() for p in paths]
        arr = (ctypes.c_char_p * len(enc))(*enc)
        h = _vp()
        check(lib().escha_ckpt_open(arr, len(enc), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().escha_ckpt_close(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass

    def projections(self) -> list:
        out = []
        for i in range(lib().escha_ckpt_num_projections(self._h)):
            info = EschaProjInfo()
            check(lib().escha_ckpt_projection(self._h, i, ctypes.byref(info)))
            out.append({"prefix": info.prefix.decode(), "K": info.K, "n_experts": info.n_experts, "in": info.n_in,
                        "out": info.n_out, "has_bias": bool(info.has_bias), "has_s_in": bool(info.has_s_in),
                        "has_s_out": bool(info.has_s_out), "has_config": bool(info.has_config),
                        "scales_all_ones": bool(info.scales_all_ones), "config_k": info.config_k})
        return out

    def tensor_info(self, name: str):
        info = EschaTensorInfo()
        check(lib().escha_ckpt_tensor_info(self._h, name.encode(), ctypes.byref(info)))
        return info.dtype.decode(), tuple(info.shape[:info.ndim]), int(info.nbytes)

    def read(self, name: str) -> np.ndarray:
        """The tensor as stored (BF16 as uint16 bit patterns), in host memory."""
        dt, shape, nbytes = self.tensor_info(name)
        a = np.empty(shape, dtype=_ST_DTYPES[dt])
        check(lib().escha_ckpt_read(self._h, name.encode(), a.ctypes.data, nbytes, 0, None))
        return a

    def load_projection(self, i: int, device="cuda", nt_major: bool = False, stream=None) -> dict:
        """Projection i's codes / rin / rout (and bias, f32) in device memory."""
        p = self.projections()[i]
        KT, NT, L = p["in"] // 16, p["out"] // 16, 16 * p["K"]
        shape = ((NT, KT, L) if nt_major else (KT, NT, L)) if not p["n_experts"] else (p["n_experts"], KT, NT, L)
        lead = (p["n_experts"],) if p["n_experts"] else ()
        codes = torch.empty(shape, dtype=torch.int16, device=device)
        rin = torch.empty(lead + (p["in"],), dtype=torch.float16, device=device)
        rout = torch.empty(lead + (p["out"],), dtype=torch.float16, device=device)
        bias = torch.empty(p["out"], dtype=torch.float32, device=device) if p["has_bias"] else None
        check(lib().escha_ckpt_load_projection(self._h, i, ptr(codes), ptr(rin), ptr(rout), ptr(bias), int(nt_major),
                                               stream_handle(stream)))
        return {"codes": codes, "rin": rin, "rout": rout, "bias": bias, "info": p}


def int8_w8a16_matvec(W, scales, x, y=None, stream=None) -> torch.Tensor:
    """y[m][o] = sum_i (scales[o] * W[o][i]) * x[m][i]; x [M][Kin] bf16/f16/f32."""
    _need_cuda(W, scales, x)
    N, Kin = W.shape
    if x.dim() == 1:
        x = x.unsqueeze(0)
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    ws_bytes = lib().int8_w8a16_workspace(N, Kin, M)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=x.device)
    check(lib().int8_w8a16_matvec(ptr(W), ptr(scales), N, Kin, ptr(x), _dtype_tag(x), M, ptr(y), ptr(ws), ws_bytes,
                                  stream_handle(stream)))
    return y


def residual_rmsnorm(h, add=None, x_out=None, eps: float = 1e-6, stream=None):
    """h f32 [T][hidden] += add (optional); then x_out (fp16 [T][hidden], made
    if None) = fp16 of the weightless RMSNorm of h. Returns x_out."""
    _need_cuda(h)
    T, H = h.shape
    if x_out is None:
        x_out = torch.empty((T, H), dtype=torch.float16, device=h.device)
    check(lib().escha_residual_rmsnorm(ptr(h), ptr(add) if add is not None else None, T, H, float(eps), ptr(x_out),
                                       stream_handle(stream)))
    return x_out


def residual_add(h, add, stream=None) -> None:
    """h += add (f32, in place) through the same kernel, without the norm."""
    _need_cuda(h, add)
    T, H = h.shape
    check(lib().escha_residual_rmsnorm(ptr(h), ptr(add), T, H, 0.0, None, stream_handle(stream)))


def int8_w8a16_dequant(W, scales, stream=None) -> torch.Tensor:
    _need_cuda(W, scales)
    N, Kin = W.shape
    out = torch.empty((N, Kin), dtype=torch.float32, device=W.device)
    check(lib().int8_w8a16_dequant(ptr(W), ptr(scales), N, Kin, ptr(out), stream_handle(stream)))
    return out


class MoeBlock:
    """Device-resident weights of one MoE block plus the C-ABI layer struct.

    ``arrays`` holds numpy arrays with the keys of ``escha_synth.moe_layer``;
    they are copied to the device once.
    """

    def __init__(self, arrays: dict, device="cuda", topk: int = 8):
        def dev(a):
            if isinstance(a, torch.Tensor):
                return a.to(device).contiguous()
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                a = a.view(np.int16)  # code words travel as raw 16-bit patterns
            return torch.from_numpy(a).to(device).contiguous()

        self.hidden = int(arrays["hidden"])
        self.inter = int(arrays["inter"])
        self.n_experts = int(arrays["n_experts"])
        self.topk = topk
        self.sh_inter = int(arrays.get("sh_inter", 0) or 0)
        self.t = {}
        self.t["router_w"] = dev(arrays["Wg"])
        self.t["gu_codes"] = dev(arrays["gu_codes"])
        self.t["gu_rin"] = dev(arrays["gu_rin"])
        self.t["gu_rout"] = dev(arrays["gu_rout"])
        self.t["dn_codes"] = dev(arrays["dn_codes"])
        self.t["dn_rin"] = dev(arrays["dn_rin"])
        self.t["dn_rout"] = dev(arrays["dn_rout"])
        self.gu_K = int(arrays["gu_codes"].shape[-1]) // 16
        self.dn_K = int(arrays["dn_codes"].shape[-1]) // 16
        if self.sh_inter:
            self.t["sh_gu_w8"] = dev(arrays["sh_gu_w8"])
            self.t["sh_gu_scale"] = dev(arrays["sh_gu_s"])
            self.t["sh_dn_w8"] = dev(arrays["sh_dn_w8"])
            self.t["sh_dn_scale"] = dev(arrays["sh_dn_s"])
            self.t["sh_gate"] = dev(arrays["sh_gate"])
        self.layer = self._struct()
        self._ws = None

    @classmethod
    def from_checkpoint(cls, ckpt: "Checkpoint", prefix: str, topk: int = 8, device="cuda", names: dict | None = None):
        """The block under ``prefix`` (e.g. "model.layers.0.mlp") of an opened
        checkpoint: stacked experts ``experts.gate_up_proj`` / ``experts.down_proj``
        (coded leaves, kt-major), router ``gate.weight``, and, when present,
        the int8 shared expert ``shared_expert.{gate_up,down}_proj.weight_int8``
        with ``weight_scale`` and its gate ``shared_expert_gate.weight``.
        ``names`` overrides any of these relative names."""
        n = {"gate_up": "experts.gate_up_proj", "down": "experts.down_proj", "router": "gate.weight",
             "sh_gu_w8": "shared_expert.gate_up_proj.weight_int8",
             "sh_gu_s": "shared_expert.gate_up_proj.weight_scale",
             "sh_dn_w8": "shared_expert.down_proj.weight_int8", "sh_dn_s": "shared_expert.down_proj.weight_scale",
             "sh_gate": "shared_expert_gate.weight"}
        n.update(names or {})
        full = {k: f"{prefix}.{v}" for k, v in n.items()}
        projs = {p["prefix"]: i for i, p in enumerate(ckpt.projections())}
        for k in ("gate_up", "down"):
            if full[k] not in projs:
                raise ValueError(f"checkpoint has no coded projection {full[k]}")
        gu = ckpt.load_projection(projs[full["gate_up"]], device=device)
        dn = ckpt.load_projection(projs[full["down"]], device=device)
        if not gu["info"]["n_experts"] or gu["info"]["n_experts"] != dn["info"]["n_experts"]:
            raise ValueError(f"{prefix}: expert projections must be stacked with one expert count")
        arrays = {"hidden": gu["info"]["in"], "inter": dn["info"]["in"], "n_experts": gu["info"]["n_experts"],
                  "Wg": ckpt.read(full["router"]),
                  "gu_codes": gu["codes"], "gu_rin": gu["rin"], "gu_rout": gu["rout"],
                  "dn_codes": dn["codes"], "dn_rin": dn["rin"], "dn_rout": dn["rout"], "sh_inter": 0}
        try:
            ckpt.tensor_info(full["sh_gu_w8"])
            has_shared = True
        except EschaError:
            has_shared = False
        if has_shared:
            arrays["sh_gu_w8"] = ckpt.read(full["sh_gu_w8"])
            arrays["sh_inter"] = arrays["sh_gu_w8"].shape[0] // 2
            arrays["sh_gu_s"] = ckpt.read(full["sh_gu_s"])
            arrays["sh_dn_w8"] = ckpt.read(full["sh_dn_w8"])
            arrays["sh_dn_s"] = ckpt.read(full["sh_dn_s"])
            arrays["sh_gate"] = ckpt.read(full["sh_gate"]).reshape(-1)
        return cls(arrays, device=device, topk=topk)

    def _struct(self) -> EschaMoeLayer:
        t = self.t
        L = EschaMoeLayer()
        L.hidden, L.inter, L.n_experts, L.topk = self.hidden, self.inter, self.n_experts, self.topk
        L.router_w = ptr(t["router_w"])
        L.gu_codes, L.gu_K, L.gu_rin, L.gu_rout = ptr(t["gu_codes"]), self.gu_K, ptr(t["gu_rin"]), ptr(t["gu_rout"])
        L.dn_codes, L.dn_K, L.dn_rin, L.dn_rout = ptr(t["dn_codes"]), self.dn_K, ptr(t["dn_rin"]), ptr(t["dn_rout"])
        L.sh_inter = self.sh_inter
        if self.sh_inter:
            L.sh_gu_w8, L.sh_gu_scale = ptr(t["sh_gu_w8"]), ptr(t["sh_gu_scale"])
            L.sh_dn_w8, L.sh_dn_scale = ptr(t["sh_dn_w8"]), ptr(t["sh_dn_scale"])
            L.sh_gate = ptr(t["sh_gate"])
        return L

    def path(self, T: int) -> int:
        """ESCHA_PATH_FUSED, ESCHA_PATH_SLOT or ESCHA_PATH_GROUPED: the kernels a
        call with T tokens runs on the current device."""
        r = lib().escha_moe_block_path(ctypes.byref(self.layer), T)
        if r < 0:
            check(r)
        return r

    def workspace(self, T: int) -> torch.Tensor:
        need = lib().escha_moe_block_workspace(ctypes.byref(self.layer), T)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.t["router_w"].device)
        return self._ws

    def __call__(self, x: torch.Tensor, out=None, ids=None, w=None, stream=None, ws=None):
        """x [T][hidden] fp16 (CUDA). Returns (out f32 [T][hidden], ids int32
        [T][topk], w f32 [T][topk]). ``ws`` optionally replaces the block's own
        workspace (e.g. one shared by the blocks of a stack)."""
        _need_cuda(x)
        T = x.shape[0]
        dev = x.device
        if out is None:
            out = torch.empty((T, self.hidden), dtype=torch.float32, device=dev)
        if ids is None:
            ids = torch.empty((T, self.topk), dtype=torch.int32, device=dev)
        if w is None:
            w = torch.empty((T, self.topk), dtype=torch.float32, device=dev)
        if ws is None:
            ws = self.workspace(T)
        check(lib().escha_moe_block(ctypes.byref(self.layer), ptr(x), T, ptr(out), ptr(ids), ptr(w), ptr(ws),
                                    ws.numel(), stream_handle(stream)))
        return out, ids, w

    def resid(self, h: torch.Tensor, add, x: torch.Tensor, eps: float = 1e-6, out=None, ids=None, w=None,
              stream=None, ws=None):
        """Residual block: h (f32 [T][hidden]) += add (or nothing when add is
        None), x (fp16 [T][hidden], written) = weightless RMSNorm of h, then the
        block on x. ``out`` may be ``add``. Returns (out, ids, w)."""
        _need_cuda(h, x)
        T = h.shape[0]
        dev = h.device
        if out is None:
            out = torch.empty((T, self.hidden), dtype=torch.float32, device=dev)
        if ids is None:
            ids = torch.empty((T, self.topk), dtype=torch.int32, device=dev)
        if w is None:
            w = torch.empty((T, self.topk), dtype=torch.float32, device=dev)
        if ws is None:
            ws = self.workspace(T)
        check(lib().escha_moe_block_resid(ctypes.byref(self.layer), ptr(h), ptr(add) if add is not None else None,
                                          float(eps), ptr(x), T, ptr(out), ptr(ids), ptr(w), ptr(ws), ws.numel(),
                                          stream_handle(stream)))
        return out, ids, w

    def route(self, x: torch.Tensor, stream=None) -> dict:
        """Diagnostic: router logits (fp16 bits), ids, w and the grouping by
        expert (counts, offsets, perm) for x [T][hidden] fp16."""
        _need_cuda(x)
        T, E, k = x.shape[0], self.n_experts, self.topk
        dev = x.device
        r = {
            "logits": torch.empty((T, E), dtype=torch.int16, device=dev),
            "ids": torch.empty((T, k), dtype=torch.int32, device=dev),
            "w": torch.empty((T, k), dtype=torch.float32, device=dev),
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "perm": torch.empty(T * k, dtype=torch.int32, device=dev),
        }
        need = lib().escha_moe_route_workspace(ctypes.byref(self.layer), T)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        check(lib().escha_moe_route(ctypes.byref(self.layer), ptr(x), T, ptr(r["logits"]), ptr(r["ids"]), ptr(r["w"]),
                                    ptr(r["counts"]), ptr(r["offsets"]), ptr(r["perm"]), ptr(ws), ws.numel(),
                                    stream_handle(stream)))
        return r


def _layer_array(blocks):
    arr = (ctypes.POINTER(EschaMoeLayer) * len(blocks))(*[ctypes.pointer(b.layer) for b in blocks])
    return arr


def seq_workspace_bytes(blocks) -> int:
    return lib().escha_moe_seq_workspace(_layer_array(blocks), len(blocks))


def blocks_path(blocks) -> int:
    """ESCHA_PATH_SLOT or ESCHA_PATH_SEQUENCE: the kernels moe_blocks runs
    these blocks on (with the route setting)."""
    r = lib().escha_moe_blocks_path(_layer_array(blocks), len(blocks))
    if r < 0:
        check(r)
    return r


def moe_blocks(blocks, xs, outs, ids=None, w=None, ws=None, stream=None, events=None):
    """Independent one-token blocks in few launches: block i of ``blocks``
    (MoeBlock) on xs[i] (fp16 [hidden] or [1][hidden]) into outs[i] (f32).
    ``ids`` / ``w``: optional lists of per-block [topk] tensors. ``ws``: a
    workspace of at least seq_workspace_bytes(blocks) bytes. ``events``: four
    torch.cuda.Event recorded between the kernels (escha_moe_blocks_timed)."""
    n = len(blocks)
    _need_cuda(*xs, *outs)
    if ws is None:
        ws = torch.empty(seq_workspace_bytes(blocks), dtype=torch.uint8, device=xs[0].device)
    px = (_vp * n)(*[ptr(t) for t in xs])
    po = (_vp * n)(*[ptr(t) for t in outs])
    pi = (_vp * n)(*[ptr(t) for t in ids]) if ids is not None else None
    pw = (_vp * n)(*[ptr(t) for t in w]) if w is not None else None
    if events is None:
        check(lib().escha_moe_blocks(_layer_array(blocks), n, px, po, pi, pw, ptr(ws), ws.numel(),
                                     stream_handle(stream)))
    else:  # four torch.cuda.Event: the kernels' boundaries (escha_moe_blocks_timed)
        ev = (_vp * 4)(*[e.cuda_event for e in events])
        check(lib().escha_moe_blocks_timed(_layer_array(blocks), n, px, po, pi, pw, ptr(ws), ws.numel(),
                                           stream_handle(stream), ev))
    return outs


class MoeStack:
    """MoE blocks on an f32 residual stream h: for each block, x =
    fp16(RMSNorm(h)) (weightless), h += block(x); the add and the norm are
    fused into the next block's call (escha_moe_block_resid). One workspace
    serves all blocks (same shapes)."""

    def __init__(self, blocks, eps: float = 1e-6):
        self.blocks = list(blocks)
        self.eps = eps
        self._ws = None
        self._seq_ws = None

    def workspace(self, T: int) -> torch.Tensor:
        need = max(lib().escha_moe_block_workspace(ctypes.byref(b.layer), T) for b in self.blocks)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.blocks[0].t["router_w"].device)
        return self._ws

    def sequence_ok(self) -> bool:
        """Whether one token runs the whole stack in one launch (escha_moe_stack)."""
        b0 = self.blocks[0]
        return (len(self.blocks) <= 48 and b0.hidden <= 2048 and b0.hidden % 256 == 0 and 2 * b0.inter // 128 <= 32
                and b0.sh_inter <= 512
                and all((b.hidden, b.inter, b.n_experts, b.topk, b.sh_inter)
                        == (b0.hidden, b0.inter, b0.n_experts, b0.topk, b0.sh_inter) for b in self.blocks))

    def __call__(self, h: torch.Tensor, x_buf=None, out_buf=None, stream=None, trace=None, sequence=False):
        """Runs the stack on h (f32 [T][hidden], updated in place). With
        ``sequence`` one token runs the whole stack in one launch
        (escha_moe_stack; same bits) when the layers allow it; by default the
        blocks run one call each (escha_moe_block_resid), measured faster for
        a dependent stack on GB300. With a list ``trace``, appends (h before
        the block, x, block output) per block as host copies (testing only: it
        synchronises; block by block)."""
        _need_cuda(h)
        T, H = h.shape
        x = x_buf if x_buf is not None else torch.empty((T, H), dtype=torch.float16, device=h.device)
        out = out_buf if out_buf is not None else torch.empty((T, H), dtype=torch.float32, device=h.device)
        if T == 1 and trace is None and sequence and self.sequence_ok():
            need = seq_workspace_bytes(self.blocks)
            if self._seq_ws is None or self._seq_ws.numel() < need:
                self._seq_ws = torch.empty(need, dtype=torch.uint8, device=h.device)
            check(lib().escha_moe_stack(_layer_array(self.blocks), len(self.blocks), ptr(h), float(self.eps), ptr(x),
                                        ptr(out), None, None, ptr(self._seq_ws), self._seq_ws.numel(),
                                        stream_handle(stream)))
            return h
        ws = self.workspace(T)
        for i, b in enumerate(self.blocks):
            b.resid(h, out if i > 0 else None, x, self.eps, out=out, stream=stream, ws=ws)
            if trace is not None:  # h after the add (the h x was normalised from), x, the block output
                trace.append([h.cpu(), x.cpu(), out.cpu()])
        residual_add(h, out, stream)
        return h
