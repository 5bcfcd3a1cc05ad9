"""Python binding of the tile-partitioned dense GEMM library (libtpgemm.so).

Argument marshalling only: every step of D = alpha*A*B + beta*C runs in the
CUDA kernels behind the C ABI of include/tpgemm.h. The functions below carry
the same names and arguments as that header; ``matmul`` is a convenience that
takes torch tensors, passes their pointers, strides and the current stream,
and allocates D with torch when none is given. There is no CPU fallback: if
the extension is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtpgemm.so")

OUT_BF16 = 0
OUT_F32 = 1
VARIANT_AUTO = 0
VARIANT_TILED = 1
VARIANT_STREAM = 2
VARIANT_EPILOGUE_ONLY = 3
VARIANT_TILED_PAIR = 4

ACT_NONE = 0
ACT_RELU = 1
ACT_SIGMOID = 2
ACT_TANH = 3

FP8_E4M3 = 0
FP8_E5M2 = 1

NVFP4 = 0
MXFP4 = 1

OK = 0
ERR_INVALID_ARG = -1
ERR_ALIGNMENT = -2
ERR_OVERLAP = -3
ERR_UNSUPPORTED_DEVICE = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6
ERR_TOO_LARGE = -7

_lib = None


class Epilogue(ctypes.Structure):
    """Mirror of struct tpgemm_epilogue (include/tpgemm.h)."""
    _fields_ = [("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int), ("activation", ctypes.c_int),
                ("aux", ctypes.c_void_p), ("ldaux", ctypes.c_int64)]


class TpgemmError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {gemm_status_string(status)} ({status})")
        self.status = status


def load_library() -> ctypes.CDLL:
    """Load libtpgemm.so from the package directory (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
        pi32, pi64 = ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int64)
        sig = {
            "gemm_create": (i32, [ctypes.POINTER(vp), i32]),
            "gemm_run": (i32, [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, f32, i32, vp]),
            "gemm_sync_status": (i32, [vp, vp]),
            "gemm_run_chunked": (i32, [vp, i32, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, f32, i32,
                                       ctypes.POINTER(vp), vp]),
            "gemm_run_batched": (i32, [vp, i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64,
                                       i64, f32, f32, i32, vp]),
            "gemm_run_grouped": (i32, [vp, i64, pi64, i64, i64, vp, i64, vp, i64, i64, vp, i64, vp, i64, f32, f32,
                                       i32, vp]),
            "gemm_run_epilogue": (i32, [vp, i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, f32, i32,
                                        ctypes.POINTER(Epilogue), vp]),
            "gemm_check_args": (i32, [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, i32]),
            "gemm_destroy": (i32, [vp]),
            "gemm_status_string": (ctypes.c_char_p, [i32]),
            "gemm_force_variant": (i32, [vp, i32]),
            "gemm_query_plan": (i32, [vp, i64, i64, i64, i32, pi32, pi32, pi32, pi64, pi32, pi32, pi32, pi32]),
            "gemm_schedule_tiles": (i64, [i64, i64, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32), i64]),
            "gemm_schedule_workers": (i32, [i64, i64, i32, i32, i32]),
            "gemm_stream_split": (i32, [i64, i64, i32, i32, pi32]),
            "gemm_tiled_ksplit": (i32, [i64, i64, i32, i32]),
            "gemm_watchdog_selftest": (i32, [vp, ctypes.c_uint64, vp]),
            "gemm_num_sms": (i32, [vp]),
            "gemm_set_workspace": (i32, [vp, vp, i64, vp]),
            "gemm_workspace_size": (i64, [vp]),
            "gemm_plan_tail_ksplit": (i32, [vp, i64, i64, i64, i32]),
            "gemm_tail_ksplit": (i32, [i32, i64, i64, i64]),
            "gemm_tail_workspace_bytes": (i64, [i64]),
            "gemm_run_noalloc": (i32, [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, f32, i32, vp,
                                       i32]),
            "gemm_run_mx": (i32, [vp, i64, i64, i64, vp, i64, i32, vp, vp, i64, i32, vp, vp, i64, vp, i64, f32, f32,
                                  i32, vp]),
            "gemm_mx_scale_bytes": (i64, [i64, i64]),
            "gemm_mx_check_args": (i32, [i64, i64, i64, vp, i64, i32, vp, vp, i64, i32, vp, vp, i64, vp, i64, f32,
                                         i32]),
            "gemm_mx_query_plan": (i32, [vp, i64, i64, i64, i32, pi32, pi32, pi64, pi32, pi32, pi32]),
            "gemm_run_fp4": (i32, [vp, i64, i64, i64, i32, vp, i64, vp, vp, i64, vp, vp, i64, vp, i64, f32, f32,
                                   i32, vp]),
            "gemm_fp4_scale_bytes": (i64, [i32, i64, i64]),
            "gemm_fp4_check_args": (i32, [i64, i64, i64, i32, vp, i64, vp, vp, i64, vp, vp, i64, vp, i64, f32,
                                          i32]),
            "gemm_fp4_query_plan": (i32, [vp, i32, i64, i64, i64, i32, pi32, pi32, pi64, pi32, pi32, pi32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


# ------------------------------------------------------------------ C ABI, same names

def gemm_create(device: int = 0) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    st = load_library().gemm_create(ctypes.byref(h), int(device))
    if st != OK:
        raise TpgemmError(st, "gemm_create")
    return h


def gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream) -> int:
    return load_library().gemm_run(h, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta,
                                   out_dtype, stream)


def gemm_run_epilogue(h, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, epi, stream) -> int:
    """epi: an Epilogue or None (plain gemm_run)."""
    return load_library().gemm_run_epilogue(h, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta,
                                            out_dtype, ctypes.byref(epi) if epi is not None else None, stream)


def gemm_run_batched(h, batch, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, D, ldd, strideD,
                     alpha, beta, out_dtype, stream) -> int:
    return load_library().gemm_run_batched(h, batch, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                                           D, ldd, strideD, alpha, beta, out_dtype, stream)


def gemm_run_grouped(h, group_rows, N, K, A, lda, B, ldb, strideB, C, ldc, D, ldd, alpha, beta, out_dtype,
                     stream) -> int:
    """group_rows: a sequence of per-group row counts (host)."""
    rows = (ctypes.c_int64 * max(len(group_rows), 1))(*[int(r) for r in group_rows])
    return load_library().gemm_run_grouped(h, len(group_rows), rows, N, K, A, lda, B, ldb, strideB, C, ldc, D, ldd,
                                           alpha, beta, out_dtype, stream)


def gemm_run_chunked(h, chunks, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, events,
                     stream) -> int:
    """events: `chunks` raw cudaEvent_t handles (e.g. torch.cuda.Event().cuda_event)."""
    ev = (ctypes.c_void_p * max(len(events), 1))(*[int(e) for e in events])
    return load_library().gemm_run_chunked(h, chunks, M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta,
                                           out_dtype, ev, stream)


def gemm_sync_status(h, stream=None) -> int:
    return load_library().gemm_sync_status(h, stream)


def gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype) -> int:
    return load_library().gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out_dtype)


def gemm_destroy(h) -> int:
    return load_library().gemm_destroy(h)


def gemm_status_string(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def gemm_force_variant(h, variant: int) -> int:
    return load_library().gemm_force_variant(h, int(variant))


def gemm_query_plan(h, M, N, K, out_dtype) -> dict:
    v, tm, tn, g, cl, sm, la = (ctypes.c_int() for _ in range(7))
    nt = ctypes.c_int64()
    st = load_library().gemm_query_plan(h, M, N, K, out_dtype, ctypes.byref(v), ctypes.byref(tm),
                                        ctypes.byref(tn), ctypes.byref(nt), ctypes.byref(g),
                                        ctypes.byref(cl), ctypes.byref(sm), ctypes.byref(la))
    if st != OK:
        raise TpgemmError(st, "gemm_query_plan")
    return dict(variant=v.value, tile_m=tm.value, tile_n=tn.value, num_tiles=nt.value, grid=g.value,
                cluster=cl.value, smem_bytes=sm.value, launches=la.value)


def gemm_schedule_workers(mt: int, nt: int, cap: int, pair: bool = False, allow_split: bool = True) -> int:
    return load_library().gemm_schedule_workers(mt, nt, cap, int(pair), int(allow_split))


def gemm_stream_split(nt: int, kb: int, mt_pad: int, num_sms: int, clusters) -> int:
    """K split (1..4) the streaming variant picks for nt panels and kb K blocks,
    given the co-resident clusters of 2, 3 and 4 CTAs."""
    arr = (ctypes.c_int32 * 3)(*[int(c) for c in clusters])
    return load_library().gemm_stream_split(nt, kb, mt_pad, num_sms, arr)


def gemm_tiled_ksplit(tiles: int, kb: int, cap2: int, cap4: int) -> int:
    """K split (1, 2 or 4) the tiled kernel picks for `tiles` 1-CTA tiles of kb K
    blocks, given the co-resident clusters of 2 and 4 CTAs."""
    return load_library().gemm_tiled_ksplit(tiles, kb, cap2, cap4)


def gemm_schedule_tiles(mt: int, nt: int, group_m: int, cap: int, worker: int, pair: bool = False,
                        allow_split: bool = True):
    """Work items (tile row, first column, width) of worker `worker`: the kernels' own schedule."""
    lib = load_library()
    n = lib.gemm_schedule_tiles(mt, nt, group_m, cap, int(pair), int(allow_split), worker, None, 0)
    if n < 0:
        raise TpgemmError(int(n), "gemm_schedule_tiles")
    buf = (ctypes.c_int32 * max(3 * n, 1))()
    lib.gemm_schedule_tiles(mt, nt, group_m, cap, int(pair), int(allow_split), worker, buf, n)
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n)]


def gemm_watchdog_selftest(h, timeout_ns: int, stream=None) -> int:
    return load_library().gemm_watchdog_selftest(h, int(timeout_ns), stream)


def gemm_num_sms(h) -> int:
    return load_library().gemm_num_sms(h)


def gemm_set_workspace(h, ws, nbytes: int, stream=None) -> int:
    """Attach (ws = device pointer) or detach (ws = None) the workspace of the
    K split of the last partial round (see include/tpgemm.h)."""
    return load_library().gemm_set_workspace(h, ws, int(nbytes), stream)


def gemm_workspace_size(h) -> int:
    return load_library().gemm_workspace_size(h)


def gemm_plan_tail_ksplit(h, M, N, K, out_dtype) -> int:
    return load_library().gemm_plan_tail_ksplit(h, M, N, K, out_dtype)


def gemm_tail_ksplit(split: int, kb: int, tail_tiles: int, ws_bytes: int) -> int:
    return load_library().gemm_tail_ksplit(split, kb, tail_tiles, ws_bytes)


def gemm_tail_workspace_bytes(tail_tiles: int) -> int:
    return load_library().gemm_tail_workspace_bytes(tail_tiles)


def gemm_run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream,
                     check_status=0) -> int:
    """gemm_run without a handle and without any device allocation, for callers
    that cannot call cudaMalloc (see include/tpgemm.h)."""
    return load_library().gemm_run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta,
                                           out_dtype, stream, int(check_status))


def gemm_run_mx(h, M, N, K, A, lda, a_format, SA, B, ldb, b_format, SB, C, ldc, D, ldd, alpha, beta, out_dtype,
                stream) -> int:
    """Block-scaled (MXFP8) GEMM; B is passed transposed ([N, K] row-major) and
    the scales in the blocked layout (see include/tpgemm.h)."""
    return load_library().gemm_run_mx(h, M, N, K, A, lda, a_format, SA, B, ldb, b_format, SB, C, ldc, D, ldd,
                                      alpha, beta, out_dtype, stream)


def gemm_mx_scale_bytes(rows: int, K: int) -> int:
    return load_library().gemm_mx_scale_bytes(rows, K)


def gemm_mx_check_args(M, N, K, A, lda, a_format, SA, B, ldb, b_format, SB, C, ldc, D, ldd, beta, out_dtype) -> int:
    return load_library().gemm_mx_check_args(M, N, K, A, lda, a_format, SA, B, ldb, b_format, SB, C, ldc, D, ldd,
                                             beta, out_dtype)


def gemm_mx_query_plan(h, M, N, K, out_dtype=OUT_BF16) -> dict:
    tm, tn, grid, cl, smem = (ctypes.c_int() for _ in range(5))
    tiles = ctypes.c_int64()
    st = load_library().gemm_mx_query_plan(h, M, N, K, out_dtype, ctypes.byref(tm), ctypes.byref(tn),
                                           ctypes.byref(tiles), ctypes.byref(grid), ctypes.byref(cl),
                                           ctypes.byref(smem))
    if st != OK:
        raise TpgemmError(st, "gemm_mx_query_plan")
    return {"tile_m": tm.value, "tile_n": tn.value, "num_tiles": tiles.value, "grid": grid.value,
            "cluster": cl.value, "smem_bytes": smem.value}


def gemm_run_fp4(h, M, N, K, fmt, A, lda, SA, B, ldb, SB, C, ldc, D, ldd, alpha, beta, out_dtype, stream) -> int:
    """Block-scaled FP4 GEMM (fmt NVFP4 or MXFP4): A [M, K/2] and B transposed
    [N, K/2] packed E2M1 bytes (lda, ldb in bytes), scales in the blocked
    layout (see include/tpgemm.h)."""
    return load_library().gemm_run_fp4(h, M, N, K, fmt, A, lda, SA, B, ldb, SB, C, ldc, D, ldd, alpha, beta,
                                       out_dtype, stream)


def gemm_fp4_scale_bytes(fmt: int, rows: int, K: int) -> int:
    return load_library().gemm_fp4_scale_bytes(fmt, rows, K)


def gemm_fp4_check_args(M, N, K, fmt, A, lda, SA, B, ldb, SB, C, ldc, D, ldd, beta, out_dtype) -> int:
    return load_library().gemm_fp4_check_args(M, N, K, fmt, A, lda, SA, B, ldb, SB, C, ldc, D, ldd, beta,
                                              out_dtype)


def gemm_fp4_query_plan(h, fmt, M, N, K, out_dtype=OUT_BF16) -> dict:
    tm, tn, grid, cl, smem = (ctypes.c_int() for _ in range(5))
    tiles = ctypes.c_int64()
    st = load_library().gemm_fp4_query_plan(h, fmt, M, N, K, out_dtype, ctypes.byref(tm), ctypes.byref(tn),
                                            ctypes.byref(tiles), ctypes.byref(grid), ctypes.byref(cl),
                                            ctypes.byref(smem))
    if st != OK:
        raise TpgemmError(st, "gemm_fp4_query_plan")
    return {"tile_m": tm.value, "tile_n": tn.value, "num_tiles": tiles.value, "grid": grid.value,
            "cluster": cl.value, "smem_bytes": smem.value}


# ------------------------------------------------------------------ torch convenience

class Gemm:
    """Owns one handle; ``__call__`` runs D = alpha*A*B + beta*C on torch tensors.

    workspace=True allocates the handle's workspace (gemm_workspace_size bytes,
    through torch) and attaches it, so that the CTA-pair kernel may split the
    last partial round over K; the constructor waits until the workspace's
    flags are clear, so the first call may go to any stream, but calls through
    this object must then not overlap on the GPU (issue them on one stream, or
    order them with events).
    """

    def __init__(self, device: int = 0, workspace: bool = False):
        self.device = int(device)
        self.handle = gemm_create(self.device)
        self._ws = None
        if workspace:
            import torch
            nbytes = gemm_workspace_size(self.handle)
            if nbytes < 0:
                raise TpgemmError(int(nbytes), "gemm_workspace_size")
            buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=f"cuda:{self.device}")
            ptr = (buf.data_ptr() + 255) // 256 * 256
            st = gemm_set_workspace(self.handle, ptr, nbytes,
                                    torch.cuda.current_stream(self.device).cuda_stream)
            if st != OK:
                raise TpgemmError(st, "gemm_set_workspace")
            # The flags are cleared on the current stream; wait for that here so
            # that calls on any stream are ordered after it.
            torch.cuda.current_stream(self.device).synchronize()
            self._ws = buf

    def close(self):
        if self.handle is not None:
            if self._ws is not None:
                import torch
                torch.cuda.synchronize(self.device)  # every call that used the workspace has finished
                gemm_set_workspace(self.handle, None, 0, None)
                self._ws = None
            gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __call__(self, A, B, C=None, alpha=1.0, beta=0.0, out_dtype=None, out=None, stream=None,
                 bias=None, activation=ACT_NONE, aux=None):
        import torch
        if out_dtype is None:
            out_dtype = out.dtype if out is not None else torch.bfloat16
        odt = {torch.bfloat16: OUT_BF16, torch.float32: OUT_F32}[out_dtype]
        M, K = A.shape
        N = B.shape[1]
        if out is None:
            out = torch.empty((M, N), dtype=out_dtype, device=A.device)
        if stream is None:
            stream = torch.cuda.current_stream(A.device).cuda_stream

        def ptr_ld(t, cols):
            if t is None:
                return None, max(cols, 1)
            if t.dim() != 2 or (t.numel() and t.stride(1) != 1):
                raise ValueError("2-D tensors with unit column stride are required")
            return t.data_ptr(), (t.stride(0) if t.shape[0] > 1 else max(t.stride(0), cols, 1))

        a, lda = ptr_ld(A, K)
        b, ldb = ptr_ld(B, N)
        c, ldc = ptr_ld(C, N)
        d, ldd = ptr_ld(out, N)
        epi = None
        if bias is not None or aux is not None or activation != ACT_NONE:
            x, ldx = ptr_ld(aux, N)
            epi = Epilogue(bias.data_ptr() if bias is not None else None,
                           OUT_F32 if (bias is not None and bias.dtype == torch.float32) else OUT_BF16,
                           int(activation), x, ldx)
        st = gemm_run_epilogue(self.handle, M, N, K, a, lda, b, ldb, c, ldc, d, ldd, float(alpha),
                               float(beta), odt, epi, stream)
        if st != OK:
            raise TpgemmError(st, "gemm_run")
        return out


_default = {}


def matmul(A, B, C=None, alpha=1.0, beta=0.0, out_dtype=None, out=None, stream=None, bias=None,
           activation=ACT_NONE, aux=None):
    """D = act(alpha*A*B + beta*C + bias) * aux on the GPU through the C ABI (one handle per device)."""
    dev = A.device.index if A.device.index is not None else 0
    if dev not in _default:
        _default[dev] = Gemm(dev)
    return _default[dev](A, B, C, alpha, beta, out_dtype, out, stream, bias, activation, aux)
