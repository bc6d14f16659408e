"""Python binding of the C-ABI: argument marshalling only; every step runs in the library.

    Y[t,:] = X[t,:] W^T + s_a (X[t,:] A_a^T) B_a^T   rows of requests naming adapter a >= 1
    Y[t,:] = X[t,:] W^T                              rows of requests naming none (id 0)

("Two 27B models on a single RTX 5090", sections 3-4.) PyTorch supplies device memory
and the CUDA stream; tensors are passed to the library as raw pointers.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib as L


class LoraError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        lib = L.load()
        super().__init__(f"{what}: {lib.lora_linear_error_string(code).decode()} ({code})")


def _check(code: int, what: str) -> None:
    if code != L.LORA_OK:
        raise LoraError(code, what)


def _i32(seq):
    seq = [int(v) for v in seq]
    return (C.c_int32 * max(1, len(seq)))(*seq), len(seq)


def _bf16_ptr(t: torch.Tensor, name: str, device: torch.device | None = None) -> int:
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, is on {t.device}")
    return t.data_ptr()


def plan(seg_offsets, seg_ids, T: int):
    """The library's planner: (fused_tiles, shrink_tiles), each a list of (row0, nrows, id)."""
    lib = L.load()
    off, n1 = _i32(seg_offsets)
    ids, n = _i32(seg_ids)
    if n1 != n + 1:
        raise ValueError("seg_offsets must hold one more entry than seg_ids")
    cap = (T + 127) // 128 + n + 1
    fused = (C.c_int32 * (3 * cap))()
    shrink = (C.c_int32 * (3 * cap))()
    nf, ns = C.c_int(cap), C.c_int(cap)
    _check(lib.lora_linear_plan(off, ids, n, T, fused, C.byref(nf), shrink, C.byref(ns)), "lora_linear_plan")
    return ([tuple(fused[3 * i:3 * i + 3]) for i in range(nf.value)],
            [tuple(shrink[3 * i:3 * i + 3]) for i in range(ns.value)])


def validate(d_in, d_out, rank, max_tokens, max_segments, x_ptr, T, seg_offsets, seg_ids, w_ptr,
             a_ptrs, b_ptrs, scales, y_ptr) -> int:
    """Run the library's host-side argument checks on raw pointers; returns the code."""
    lib = L.load()
    off, _ = _i32(seg_offsets)
    ids, n = _i32(seg_ids)
    na = len(a_ptrs)
    A = (C.c_void_p * max(1, na))(*[p for p in a_ptrs])
    B = (C.c_void_p * max(1, na))(*[p for p in b_ptrs])
    S = (C.c_float * max(1, na))(*[float(s) for s in scales])
    return lib.lora_linear_validate(d_in, d_out, rank, max_tokens, max_segments, x_ptr, T,
                                    off if seg_offsets is not None else None,
                                    ids if seg_ids is not None else None, n, w_ptr,
                                    A if a_ptrs is not None else None, B if b_ptrs is not None else None,
                                    S if scales is not None else None, na, y_ptr)


def launch_shape(d_in, d_out, rank, num_sms, T, seg_offsets, seg_ids, w4=False) -> dict:
    """The launch shape ``forward`` (or ``forward_w4``) would choose for these rows on a GPU with
    ``num_sms`` SMs, computed by the library on the host alone (no device needed)."""
    lib = L.load()
    off, _ = _i32(seg_offsets)
    ids, n = _i32(seg_ids)
    v = [C.c_int() for _ in range(7)]
    _check(lib.lora_linear_shape(d_in, d_out, rank, num_sms, T, off, ids, n, int(bool(w4)),
                                 *[C.byref(x) for x in v]),
           "lora_linear_shape")
    return dict(zip(("cluster", "tile_n", "bk", "stages", "unit_order", "fused_units", "shrink_units"),
                    [x.value for x in v]))


def k_split(d_in, d_out, rank, max_tokens, num_sms) -> int:
    """The K split (1 or 2) a handle of this shape and max_tokens chooses at create on a GPU
    with ``num_sms`` SMs, computed by the library on the host alone."""
    lib = L.load()
    v = C.c_int()
    _check(lib.lora_linear_k_split(d_in, d_out, rank, max_tokens, num_sms, C.byref(v)), "lora_linear_k_split")
    return v.value


def host_chunks(T) -> list:
    """Row bounds of the chunks ``forward_host`` runs T rows in (0 first, T last)."""
    lib = L.load()
    bounds = (C.c_int32 * 17)()
    n = C.c_int()
    _check(lib.lora_linear_host_chunks(T, bounds, C.byref(n)), "lora_linear_host_chunks")
    return [bounds[i] for i in range(n.value + 1)]


def w4_repack(src: torch.Tensor, dst: torch.Tensor | None = None,
              stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """4-bit base weight, plain layout (uint8 [d_out, d_in/2], low nibble = even input,
    two's complement) -> the kernel layout that ``forward_w4`` reads. ``dst`` may be ``src``."""
    lib = L.load()
    if src.dtype != torch.uint8 or not src.is_contiguous() or src.device.type != "cuda":
        raise TypeError("src must be a contiguous uint8 CUDA tensor")
    if dst is None:
        dst = torch.empty_like(src)
    if dst.dtype != torch.uint8 or not dst.is_contiguous() or dst.device != src.device or dst.numel() != src.numel():
        raise TypeError("dst must be a contiguous uint8 tensor of src's size on src's device")
    s = stream if stream is not None else torch.cuda.current_stream(src.device)
    with torch.cuda.device(src.device):
        _check(lib.lora_linear_w4_repack(src.data_ptr(), dst.data_ptr(), src.numel(), C.c_void_p(s.cuda_stream)),
               "lora_linear_w4_repack")
    return dst


class LoraLinear:
    """One handle: a projection shape (d_in -> d_out, rank r) on one CUDA device."""

    def __init__(self, d_in: int, d_out: int, rank: int, max_tokens: int, max_segments: int = 64,
                 device: int | torch.device | None = None):
        self._lib = L.load()
        if device is None:
            device = torch.cuda.current_device()
        if isinstance(device, torch.device):
            device = device.index if device.index is not None else torch.cuda.current_device()
        self.device = torch.device("cuda", int(device))
        self.d_in, self.d_out, self.rank = d_in, d_out, rank
        self.max_tokens, self.max_segments = max_tokens, max_segments
        h = C.c_void_p()
        _check(self._lib.lora_linear_create(C.byref(h), d_in, d_out, rank, max_tokens, max_segments,
                                            int(device)), "lora_linear_create")
        self._h = h

    # ------------------------------------------------------------------ lifecycle
    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.lora_linear_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ------------------------------------------------------------------ marshalling
    def _adapters(self, A, B, scales):
        na = len(A)
        if len(B) != na or len(scales) != na:
            raise ValueError("A, B and scales must have one entry per adapter")
        a_arr = (C.c_void_p * max(1, na))(*[_bf16_ptr(a, "A", self.device) if a is not None else None for a in A])
        b_arr = (C.c_void_p * max(1, na))(*[_bf16_ptr(b, "B", self.device) if b is not None else None for b in B])
        s_arr = (C.c_float * max(1, na))(*[float(s) for s in scales])
        return a_arr, b_arr, s_arr, na

    def forward(self, x: torch.Tensor, seg_offsets, seg_ids, W: torch.Tensor, A, B, scales,
                y: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """Y for the batch x [T, d_in]; enqueued on `stream` (default: the current stream)."""
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.d_out), dtype=torch.bfloat16, device=self.device)
        off, _ = _i32(seg_offsets)
        ids, n = _i32(seg_ids)
        a_arr, b_arr, s_arr, na = self._adapters(A, B, scales)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        rc = self._lib.lora_linear_forward(self._h, _bf16_ptr(x, "x", self.device), T, off, ids, n,
                                           _bf16_ptr(W, "W", self.device), a_arr, b_arr, s_arr, na,
                                           _bf16_ptr(y, "y", self.device), C.c_void_p(s.cuda_stream))
        _check(rc, "lora_linear_forward")
        return y

    def forward_w4(self, x: torch.Tensor, seg_offsets, seg_ids, Wq: torch.Tensor, Ws: torch.Tensor, A, B, scales,
                   y: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """Same with a 4-bit base: Wq uint8 [d_out, d_in/2] in the kernel layout (``w4_repack`` of
        the plain layout), Ws bf16 [d_in/128, d_out]; W[n,k] = q[n,k] * Ws[k//128, n]."""
        if Wq.dtype != torch.uint8 or not Wq.is_contiguous() or Wq.device != self.device:
            raise TypeError("Wq must be a contiguous uint8 tensor on the handle's device")
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.d_out), dtype=torch.bfloat16, device=self.device)
        off, _ = _i32(seg_offsets)
        ids, n = _i32(seg_ids)
        a_arr, b_arr, s_arr, na = self._adapters(A, B, scales)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        rc = self._lib.lora_linear_forward_w4(self._h, _bf16_ptr(x, "x", self.device), T, off, ids, n,
                                              Wq.data_ptr(), _bf16_ptr(Ws, "Ws", self.device), a_arr, b_arr, s_arr,
                                              na, _bf16_ptr(y, "y", self.device), C.c_void_p(s.cuda_stream))
        _check(rc, "lora_linear_forward_w4")
        return y

    def forward_host_w4(self, x_host: torch.Tensor, seg_offsets, seg_ids, Wq: torch.Tensor, Ws: torch.Tensor, A, B,
                        scales, y_host: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """forward_w4 from and to host bf16 tensors; waits for completion."""
        if x_host.device.type != "cpu" or y_host.device.type != "cpu":
            raise ValueError("forward_host_w4 takes host tensors")
        if Wq.dtype != torch.uint8 or not Wq.is_contiguous() or Wq.device != self.device:
            raise TypeError("Wq must be a contiguous uint8 tensor on the handle's device")
        T = x_host.shape[0]
        off, _ = _i32(seg_offsets)
        ids, n = _i32(seg_ids)
        a_arr, b_arr, s_arr, na = self._adapters(A, B, scales)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        rc = self._lib.lora_linear_forward_host_w4(self._h, _bf16_ptr(x_host, "x"), T, off, ids, n, Wq.data_ptr(),
                                                   _bf16_ptr(Ws, "Ws", self.device), a_arr, b_arr, s_arr, na,
                                                   _bf16_ptr(y_host, "y"), C.c_void_p(s.cuda_stream))
        _check(rc, "lora_linear_forward_host_w4")
        return y_host

    def forward_host(self, x_host: torch.Tensor, seg_offsets, seg_ids, W: torch.Tensor, A, B, scales,
                     y_host: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
        """Same, from and to host bf16 tensors (pinned for speed); waits for completion."""
        if x_host.device.type != "cpu" or y_host.device.type != "cpu":
            raise ValueError("forward_host takes host tensors")
        T = x_host.shape[0]
        off, _ = _i32(seg_offsets)
        ids, n = _i32(seg_ids)
        a_arr, b_arr, s_arr, na = self._adapters(A, B, scales)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        rc = self._lib.lora_linear_forward_host(self._h, _bf16_ptr(x_host, "x"), T, off, ids, n,
                                                _bf16_ptr(W, "W", self.device), a_arr, b_arr, s_arr, na,
                                                _bf16_ptr(y_host, "y"), C.c_void_p(s.cuda_stream))
        _check(rc, "lora_linear_forward_host")
        return y_host

    # ------------------------------------------------------------------ diagnostics
    def status(self, reset: bool = False) -> int:
        return self._lib.lora_linear_status(self._h, 1 if reset else 0)

    def set_option(self, option: int, value: int) -> None:
        _check(self._lib.lora_linear_set_option(self._h, option, int(value)), "lora_linear_set_option")

    def timing(self, kind: int):
        ms, n, allc = C.c_double(), C.c_longlong(), C.c_longlong()
        _check(self._lib.lora_linear_timing(self._h, kind, C.byref(ms), C.byref(n), C.byref(allc)),
               "lora_linear_timing")
        return ms.value, n.value, allc.value

    def describe(self, T, seg_offsets, seg_ids) -> dict:
        off, _ = _i32(seg_offsets)
        ids, n = _i32(seg_ids)
        v = [C.c_int() for _ in range(7)]
        _check(self._lib.lora_linear_describe(self._h, T, off, ids, n, *[C.byref(x) for x in v]),
               "lora_linear_describe")
        return dict(zip(("tile_n", "n_tiles", "n_units", "grid", "stages", "has_shrink", "unit_order"),
                        [x.value for x in v]))
