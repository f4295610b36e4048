"""GB300 (sm_103a) heterogeneous multi-LoRA delta: y_i += s_k (x_i A_k) B_k over a
batch whose rows are grouped by adapter id, with paged adapter storage, released
rows skipped, and an in-place merge / unmerge of W +/- s A B.

Every step runs in the CUDA kernels of ``liblora.so`` behind the C ABI declared in
``include/lora.h``; this module only marshals torch tensors (device memory and
streams) and numpy id arrays into those calls, under the same names.  Importing it
without the built library raises: there is no other implementation.
"""
from __future__ import annotations

import ctypes
import weakref

import numpy as np
import torch

from . import _lib

__all__ = ["LoraError", "Context", "AdapterTable", "lora_plan_build", "lora_shrink",
           "lora_expand", "lora_fused", "lora_fused_noalloc", "lora_base_fused", "PreparedFused", "PreparedFusedDeviceIds", "lora_merge", "lora_unmerge", "lora_page_in", "lora_fused_device_ids", "lora_tune_shape",
           "KIND_ROWS_FUSED", "KIND_SHRINK", "KIND_EXPAND", "KIND_TILE_FUSED", "KIND_MERGE",
           "OPT_TILE_PATH", "OPT_MERGE_KERNEL", "OPT_TILE_MIN_RUN", "OPT_EARLY_PAGES", "OPT_DEVICE_PLAN",
           "OPT_EARLY_INPUT", "OPT_ROWS_B_OVER_A",
           "library_path"]

KIND_ROWS_FUSED, KIND_SHRINK, KIND_EXPAND, KIND_TILE_FUSED, KIND_MERGE = range(5)
OPT_TILE_PATH, OPT_MERGE_KERNEL, OPT_TILE_MIN_RUN, OPT_EARLY_PAGES, OPT_DEVICE_PLAN = 1, 2, 3, 4, 5
OPT_EARLY_INPUT = 6
OPT_ROWS_B_OVER_A = 7
ERROR_NAMES = {0: "LORA_OK", -1: "LORA_E_INVAL", -2: "LORA_E_RANK", -3: "LORA_E_ADAPTER",
               -4: "LORA_E_NOT_RESIDENT", -5: "LORA_E_PAGE", -6: "LORA_E_CUDA",
               -7: "LORA_E_TIMEOUT", -8: "LORA_E_NOMEM", -9: "LORA_E_CAPACITY",
               -10: "LORA_E_UNSUPPORTED", -11: "LORA_E_IO", -12: "LORA_E_NOTUNED"}

_L = _lib.load()


def library_path() -> str:
    return _lib.LIB_PATH


class LoraError(RuntimeError):
    def __init__(self, code: int, detail: str = ""):
        self.code = code
        self.name = ERROR_NAMES.get(code, str(code))
        msg = f"{self.name}: {_L.lora_strerror(code).decode()}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def _check(rc: int, ctx: "Context | None" = None) -> int:
    if rc < 0:
        detail = ""
        if rc == -6 and ctx is not None and ctx.handle:
            detail = (_L.lora_last_cuda_error(ctx.handle) or b"").decode()
        raise LoraError(rc, detail)
    return rc


def _stream(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: torch.Tensor, what: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    return t.data_ptr()


def _ids(ids):
    """(int32 contiguous array, its address, length)."""
    if not (isinstance(ids, np.ndarray) and ids.dtype == np.int32 and ids.flags.c_contiguous):
        ids = np.ascontiguousarray(np.asarray(ids), dtype=np.int32)
    if ids.ndim != 1:
        raise ValueError("ids must be one-dimensional")
    return ids, ids.__array_interface__["data"][0], ids.shape[0]


def _rows(t: torch.Tensor, what: str):
    """(pointer, row stride in elements, columns) of a 2-D row-major 16-bit CUDA tensor."""
    st = t.stride()
    if len(st) != 2 or st[1] != 1 or t.element_size() != 2 or not t.is_cuda:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{what} must be a CUDA tensor")
        raise ValueError(f"{what} must be a 2-D row-major bf16 tensor")
    return t.data_ptr(), st[0], t.shape[1]


class Context:
    """A library context on one device (plan staging buffers, status word, tile table)."""

    def __init__(self, device: int = 0, max_rows: int = 1 << 16, max_rank: int = 64):
        """device = -1: host-only context (plans and tile tables, no launches)."""
        if isinstance(device, int) and device < 0:
            self.device, idx = None, -1
        else:
            self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
            idx = self.device.index or 0
        h = ctypes.c_void_p()
        self.handle = None
        self._tables = weakref.WeakSet()
        _check(_L.lora_ctx_create(idx, int(max_rows), int(max_rank), ctypes.byref(h)))
        self.handle = h.value

    def close(self):
        """Destroy the context and every table registered with it."""
        if self.handle:
            for t in list(self._tables):
                t.close()
            _L.lora_ctx_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def tiles_load(self, path: str):
        _check(_L.lora_tiles_load(self.handle, path.encode()), self)

    def tiles_save(self, path: str):
        _check(_L.lora_tiles_save(self.handle, path.encode()), self)

    def tiles_count(self) -> int:
        return int(_L.lora_tiles_count(self.handle))

    def tile_status(self) -> str:
        """"LORA_OK" if the last call found all its launch shapes in the tile table,
        "LORA_E_NOTUNED" if it took a built-in default for one of them."""
        return ERROR_NAMES[int(_L.lora_tile_status(self.handle))]

    def tune(self, shapes_path: str, out_path: str | None = None, stream=None):
        """lora_tune: the offline search over a shape file (see include/lora.h); the
        winners go into this context's table, and to out_path if given."""
        _check(_L.lora_tune(self.handle, shapes_path.encode(),
                            out_path.encode() if out_path else None,
                            _stream(stream, self.device) if self.device is not None else None),
               self)

    def sync_status(self, stream=None) -> int:
        """Synchronize and read back the device status word (raises on a timeout)."""
        return _check(_L.lora_sync_status(self.handle, _stream(stream, self.device)), self)

    def selftest_timeout(self, limit_us: int = 10000, stream=None):
        """Launch a bounded wait that runs out (see include/lora.h): the next
        sync_status raises LORA_E_TIMEOUT and the context stays usable."""
        _check(_L.lora_selftest_timeout(self.handle, int(limit_us), _stream(stream, self.device)), self)

    def set_option(self, option: int, value: int):
        """LORA_OPT_* (see include/lora.h): OPT_TILE_PATH, OPT_MERGE_KERNEL,
        OPT_TILE_MIN_RUN, OPT_EARLY_PAGES, OPT_DEVICE_PLAN, OPT_EARLY_INPUT,
        OPT_ROWS_B_OVER_A."""
        _check(_L.lora_ctx_set_option(self.handle, int(option), int(value)), self)

    def profile_begin(self, every: int = 1):
        """Start bracketing every `every`-th kernel launch with CUDA events."""
        _check(_L.lora_profile_begin(self.handle, int(every)), self)

    def profile_end(self):
        """Stop; returns {family: (device ms, launches)} for the row-gather, tile shrink,
        merge and streaming expand kernels: every launch made while profiling, and
        their device time (the bracketed launches' mean times that count)."""
        ms = (ctypes.c_double * 5)()
        n = (ctypes.c_int64 * 5)()
        _check(_L.lora_profile_end(self.handle, ms, n), self)
        return {name: (ms[i], int(n[i]))
                for i, name in enumerate(("rows", "shrink", "merge", "expand", "proj"))}

    def launch_count(self) -> int:
        """Kernels launched by this context so far."""
        return int(_L.lora_launch_count(self.handle))

    def last_path(self):
        """(path bits, launches) of the last call: 1 row-gather, 2 tensor-core tile,
        4 merge."""
        n = ctypes.c_int()
        p = _L.lora_last_path(self.handle, ctypes.byref(n))
        return p, n.value


class AdapterTable:
    """Registered adapter table over caller-owned device pools of bf16 pages.

    a_pool / b_pool: CUDA tensors [n_pages, page_width] (bf16 or 16-bit ints); may be
    the same tensor.  rank, scale: [n_adapters]; a_pages, b_pages: [n_adapters,
    max_rank] page ids (-1 = not resident).  The pools are kept referenced here so
    they outlive the table."""

    def __init__(self, ctx: Context, a_pool: torch.Tensor, b_pool: torch.Tensor, rank, scale,
                 a_pages, b_pages):
        self.ctx = ctx
        self.a_pool, self.b_pool = a_pool, b_pool
        for t, nm in ((a_pool, "a_pool"), (b_pool, "b_pool")):
            if t.dim() != 2 or t.element_size() != 2 or not t.is_contiguous():
                raise ValueError(f"{nm} must be a contiguous 2-D 16-bit tensor")
        self.rank = np.ascontiguousarray(rank, dtype=np.int32)
        self.scale = np.ascontiguousarray(scale, dtype=np.float32)
        self.a_pages = np.ascontiguousarray(a_pages, dtype=np.int32)
        self.b_pages = np.ascontiguousarray(b_pages, dtype=np.int32)
        n_adapters, max_rank = self.a_pages.shape
        self.n_adapters, self.max_rank = n_adapters, max_rank
        h = ctypes.c_void_p()
        if ctx.device is None:      # host-only context: pools are never dereferenced
            pa, pb = a_pool.data_ptr(), b_pool.data_ptr()
        else:
            pa, pb = _dev_ptr(a_pool, "a_pool"), _dev_ptr(b_pool, "b_pool")
        _check(_L.lora_table_create(
            ctx.handle, pa, a_pool.shape[0], a_pool.shape[1],
            pb, b_pool.shape[0], b_pool.shape[1], n_adapters, max_rank,
            self.rank.ctypes.data, self.scale.ctypes.data, self.a_pages.ctypes.data,
            self.b_pages.ctypes.data, ctypes.byref(h)), ctx)
        self.handle = h.value
        ctx._tables.add(self)

    def invalidate(self, adapter: int = -1):
        """The pages of `adapter` (-1: every adapter) were written outside lora_page_in:
        the table's dense copy of them is stale (see include/lora.h)."""
        _check(_L.lora_table_invalidate(self.handle, int(adapter)))

    def close(self):
        if getattr(self, "handle", None):
            _L.lora_table_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def lora_plan_build(ctx: Context, table: AdapterTable, ids) -> dict:
    """Host-side grouping of one batch (copies of the context's plan arrays)."""
    ids, pid, n = _ids(ids)
    v = _lib.PlanView()
    _check(_L.lora_plan_build(ctx.handle, table.handle, pid, n, ctypes.byref(v)), ctx)

    def arr(p, n):
        return np.ctypeslib.as_array(p, shape=(n,)).copy() if n > 0 else np.zeros(0, np.int32)
    return {"active_rows": arr(v.active_rows, v.n_active), "perm": arr(v.perm, v.n_active),
            "seg_offsets": arr(v.seg_offsets, v.n_segments + 1),
            "seg_adapter": arr(v.seg_adapter, v.n_segments),
            "row_items": int(v.row_items), "tile_items": int(v.tile_items),
            "rows_per_item": int(v.rows_per_item), "tile_min_run": int(v.tile_min_run)}


def lora_shrink(ctx: Context, table: AdapterTable, ids, x: torch.Tensor, v: torch.Tensor,
                stream=None):
    """v[i, :r_k] = x_i A_k (fp32) for rows with ids[i] >= 0."""
    ids, pid, n = _ids(ids)
    px, ldx, d_in = _rows(x, "x")
    if v.dtype != torch.float32 or v.dim() != 2 or v.stride(1) != 1:
        raise ValueError("v must be a 2-D row-major float32 tensor")
    _check(_L.lora_shrink(ctx.handle, table.handle, pid, n, px, ldx, d_in, _dev_ptr(v, "v"),
                          v.stride(0), _stream(stream, ctx.device)), ctx)


def lora_expand(ctx: Context, table: AdapterTable, ids, v: torch.Tensor, y: torch.Tensor,
                stream=None):
    """y_i <- bf16(y_i + s_k v_i B_k) in place for rows with ids[i] >= 0."""
    ids, pid, n = _ids(ids)
    py, ldy, d_out = _rows(y, "y")
    if v.dtype != torch.float32 or v.dim() != 2 or v.stride(1) != 1:
        raise ValueError("v must be a 2-D row-major float32 tensor")
    _check(_L.lora_expand(ctx.handle, table.handle, pid, n, _dev_ptr(v, "v"), v.stride(0), py,
                          ldy, d_out, _stream(stream, ctx.device)), ctx)


def lora_fused(ctx: Context, table: AdapterTable, ids, x: torch.Tensor, y: torch.Tensor,
               stream=None):
    """y_i <- bf16(y_i + s_k (x_i A_k) B_k) in place for rows with ids[i] >= 0."""
    ids, pid, n = _ids(ids)
    px, ldx, d_in = _rows(x, "x")
    py, ldy, d_out = _rows(y, "y")
    rc = _L.lora_fused(ctx.handle, table.handle, pid, n, px, ldx, d_in, py, ldy, d_out,
                       _stream(stream, ctx.device))
    if rc:
        _check(rc, ctx)


def lora_fused_device_ids(ctx: Context, table: AdapterTable, ids: torch.Tensor, x: torch.Tensor,
                          y: torch.Tensor, stream=None):
    """lora_fused with the ids in device memory (a CUDA int32 tensor [n], -1 =
    released): planned on the GPU, nothing read on the host, graph-capturable.  An
    id the table cannot serve leaves its row unchanged and shows up as
    LORA_E_ADAPTER at the next sync_status (see include/lora.h)."""
    if not isinstance(ids, torch.Tensor) or not ids.is_cuda or ids.dtype != torch.int32 or \
            ids.dim() != 1 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous 1-D int32 CUDA tensor")
    px, ldx, d_in = _rows(x, "x")
    py, ldy, d_out = _rows(y, "y")
    _check(_L.lora_fused_device_ids(ctx.handle, table.handle, ids.data_ptr(), ids.shape[0], px,
                                    ldx, d_in, py, ldy, d_out, _stream(stream, ctx.device)), ctx)


def lora_base_fused(ctx: Context, table: AdapterTable, ids, x: torch.Tensor, W: torch.Tensor,
                    y: torch.Tensor, stream=None):
    """y_i <- bf16(x_i W + s_k (x_i A_k) B_k) (x_i W alone for ids[i] == -1): the base
    projection with the adapter term in one tensor-core GEMM; y is written, not read.
    W is [d_in, d_out] row-major."""
    ids, pid, n = _ids(ids)
    px, ldx, d_in = _rows(x, "x")
    pw, ldw, d_out = _rows(W, "W")
    py, ldy, d_out_y = _rows(y, "y")
    if W.shape[0] != d_in or d_out_y != d_out:
        raise ValueError("shapes: x [n, d_in], W [d_in, d_out], y [n, d_out]")
    _check(_L.lora_base_fused(ctx.handle, table.handle, pid, n, px, ldx, d_in, pw, ldw, py, ldy,
                              d_out, _stream(stream, ctx.device)), ctx)


def lora_fused_noalloc(ctx: Context, table: AdapterTable, ids, x: torch.Tensor, y: torch.Tensor,
                       stream=None):
    """lora_fused for callers that must not allocate while it runs: its scratch is
    fixed device arrays inside the library (12 MB: 4 MB of partial V and 8 MB of
    dense adapter rows, committed when a context is created); raises
    LORA_E_CAPACITY beyond their limits (see include/lora.h)."""
    ids, pid, n = _ids(ids)
    px, ldx, d_in = _rows(x, "x")
    py, ldy, d_out = _rows(y, "y")
    _check(_L.lora_fused_noalloc(ctx.handle, table.handle, pid, n, px, ldx, d_in, py, ldy, d_out,
                                 _stream(stream, ctx.device)), ctx)


class _PreparedCall:
    """A fused call with fixed x, y, table and stream (a decode loop's persistent
    buffers).  The marshalling happens once: for each ids object among the last 256
    it was handed, a filled lora_fused_args block is kept, and a call passes only
    that block's address.  Only the object is recognised, never its contents: the
    library reads the ids on every call."""

    _KEEP = 256
    _ENTRY = ""

    def __init__(self, ctx: Context, table: AdapterTable, x: torch.Tensor, y: torch.Tensor,
                 stream=None):
        px, ldx, d_in = _rows(x, "x")
        py, ldy, d_out = _rows(y, "y")
        self._keep = (ctx, table, x, y)
        self._ctx = ctx
        self._fn = _lib.untyped(self._ENTRY)
        self._fields = dict(ctx=ctx.handle, table=table.handle, x=px, ldx=ldx, d_in=d_in, y=py,
                            ldy=ldy, d_out=d_out, stream=_stream(stream, ctx.device))
        # id(ids object) -> (the object, kept alive so its id stays its own; its
        # argument block; the block's address)
        self._seen = {}

    def _ids_ptr(self, ids):
        raise NotImplementedError

    def _block(self, ids):
        ptr, n, keep = self._ids_ptr(ids)
        blk = _lib.FusedArgs(ids=ptr, n=n, **self._fields)
        ref = ctypes.byref(blk)
        if keep:
            if len(self._seen) >= self._KEEP:
                self._seen.pop(next(iter(self._seen)))
            self._seen[id(ids)] = (ids, blk, ref)
        return blk, ref

    def bind(self, ids):
        """Convert and keep the arguments for this ids object without launching, so
        that the first call with it costs no more than the later ones."""
        self._block(ids)

    def __call__(self, ids):
        hit = self._seen.get(id(ids))
        if hit is not None and hit[0] is ids:
            rc = self._fn(hit[2])
        else:
            blk, ref = self._block(ids)
            rc = self._fn(ref)
        if rc:
            _check(rc, self._ctx)


class PreparedFused(_PreparedCall):
    """lora_fused with fixed x, y, table and stream; call it with the host ids
    (int32 array, -1 = released).  An array used as it is (int32, contiguous) is
    remembered, so a persistent ids buffer rewritten in place between steps, or a
    ring of them, costs little more than the C function itself."""

    _ENTRY = "lora_fused_args_call"

    def _ids_ptr(self, ids):
        arr, pid, n = _ids(ids)
        return pid, n, arr is ids


class PreparedFusedDeviceIds(_PreparedCall):
    """lora_fused_device_ids with fixed x, y, table and stream; call it with the ids
    as a contiguous 1-D int32 CUDA tensor (its data pointer and length are taken when
    the tensor is first seen)."""

    _ENTRY = "lora_fused_device_ids_args_call"

    def _ids_ptr(self, ids):
        if not isinstance(ids, torch.Tensor) or not ids.is_cuda or ids.dtype != torch.int32 or \
                ids.dim() != 1 or not ids.is_contiguous():
            raise ValueError("ids must be a contiguous 1-D int32 CUDA tensor")
        return ids.data_ptr(), ids.shape[0], True


def lora_merge(ctx: Context, table: AdapterTable, adapter: int, W: torch.Tensor, stream=None):
    """W <- bf16(W + s_k A_k B_k) in place (W is [d_in, d_out] row-major)."""
    pw, ldw, d_out = _rows(W, "W")
    _check(_L.lora_merge(ctx.handle, table.handle, int(adapter), pw, ldw, W.shape[0], d_out,
                         _stream(stream, ctx.device)), ctx)


def lora_unmerge(ctx: Context, table: AdapterTable, adapter: int, W: torch.Tensor, stream=None):
    """W <- bf16(W - s_k A_k B_k) in place."""
    pw, ldw, d_out = _rows(W, "W")
    _check(_L.lora_unmerge(ctx.handle, table.handle, int(adapter), pw, ldw, W.shape[0], d_out,
                           _stream(stream, ctx.device)), ctx)


def lora_page_in(ctx: Context, table: AdapterTable, adapter: int, host_a: torch.Tensor,
                 host_b: torch.Tensor, stream=None):
    """Copy adapter `adapter`'s A and B into its pages of the table's pools, on
    `stream` (asynchronous).  host_a: [rank, d_in] and host_b: [rank, d_out] bf16 (or
    their 16-bit images) in page-locked CPU memory, contiguous; row j of host_a is
    column j of A_k, row j of host_b is row j of B_k.  Keep both alive and unchanged
    until the stream has passed the call (see include/lora.h)."""
    r = int(table.rank[int(adapter)]) if 0 <= int(adapter) < table.n_adapters else -1
    for name, h in (("host_a", host_a), ("host_b", host_b)):
        if not isinstance(h, torch.Tensor) or h.device.type != "cpu" or not h.is_pinned():
            raise ValueError(f"{name} must be a page-locked CPU tensor")
        if h.dim() != 2 or not h.is_contiguous() or h.element_size() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D 16-bit tensor")
        if r >= 0 and h.shape[0] != r:
            raise ValueError(f"{name} has {h.shape[0]} rows, adapter {adapter} has rank {r}")
    _check(_L.lora_page_in(ctx.handle, table.handle, int(adapter), host_a.data_ptr(),
                           host_a.shape[1], host_b.data_ptr(), host_b.shape[1],
                           _stream(stream, ctx.device)), ctx)


def lora_tune_shape(ctx: Context, table: AdapterTable, kind: int, ids, x: torch.Tensor,
                    y: torch.Tensor, iters: int = 20, stream=None) -> float:
    """Offline search for one shape (see include/lora.h); returns the best time in us
    and keeps the winning configuration in the context's table.  For KIND_MERGE, x is
    W, y is ignored and ids[0] is the adapter."""
    ids, pid, n = _ids(ids)
    px, ldx, d_in = _rows(x, "x")
    if kind == KIND_MERGE:
        py, ldy, d_out = px, ldx, d_in
        d_in = x.shape[0]
    else:
        py, ldy, d_out = _rows(y, "y")
    best = ctypes.c_float()
    _check(_L.lora_tune_shape(ctx.handle, table.handle, int(kind), pid, n, px, ldx, d_in, py,
                              ldy, d_out, int(iters),
                              ctypes.byref(best), _stream(stream, ctx.device)), ctx)
    return float(best.value)
