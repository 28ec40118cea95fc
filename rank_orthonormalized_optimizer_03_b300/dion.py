"""ctypes binding of libdion.so (declared in include/dion.h).

Argument marshalling only: every step of the optimizer runs in the library's
CUDA kernels.  PyTorch provides device memory (the caller's tensors and the
workspace) and the current CUDA stream.  There is no fallback: if the shared
library is missing or cannot be loaded, importing :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdion.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
HEADER = os.path.join(INCLUDE, "dion.h")

DION_OK, DION_ERR_INVALID_ARG, DION_ERR_CUDA, DION_ERR_WORKSPACE, DION_ERR_UNSUPPORTED = range(5)
DION_MAT_OK, DION_MAT_CHOL_BREAKDOWN, DION_MAT_NONFINITE, DION_MAT_TIMEOUT, DION_MAT_SHIFTED = 0, 1, 2, 4, 8
# bits that mean the matrix was not updated (DION_MAT_SHIFTED is informational)
FATAL = DION_MAT_CHOL_BREAKDOWN | DION_MAT_NONFINITE | DION_MAT_TIMEOUT
VARIANT = {"dion": 0, "orth": 1, "lowrank_muon": 2}
DTYPE_F32, DTYPE_BF16 = 0, 1
BUF_P, BUF_U, BUF_W = 0, 1, 2


class MatrixDesc(ctypes.Structure):
    _fields_ = [
        ("X", ctypes.c_void_p), ("G", ctypes.c_void_p), ("R", ctypes.c_void_p), ("V", ctypes.c_void_p),
        ("m", ctypes.c_int64), ("n", ctypes.c_int64), ("r", ctypes.c_int64),
        ("ld_x", ctypes.c_int64), ("ld_g", ctypes.c_int64), ("ld_r", ctypes.c_int64),
        ("g_dtype", ctypes.c_int32), ("variant", ctypes.c_int32),
        ("eta", ctypes.c_float), ("beta", ctypes.c_float), ("scale", ctypes.c_float),
        ("reserved", ctypes.c_float),
    ]


class MuonDesc(ctypes.Structure):
    _fields_ = [
        ("X", ctypes.c_void_p), ("G", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("m", ctypes.c_int64), ("n", ctypes.c_int64),
        ("ld_x", ctypes.c_int64), ("ld_g", ctypes.c_int64), ("ld_b", ctypes.c_int64),
        ("g_dtype", ctypes.c_int32), ("eta", ctypes.c_float), ("mu", ctypes.c_float), ("scale", ctypes.c_float),
    ]


MUON_PRECISION = {"bf16": 0, "tf32": 1, "fp32": 2}


class DionError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}: {detail}")
        self.code = code


STATUS_NAMES = {0: "DION_OK", 1: "DION_ERR_INVALID_ARG", 2: "DION_ERR_CUDA",
                3: "DION_ERR_WORKSPACE", 4: "DION_ERR_UNSUPPORTED"}

_lib = None


def _declare(L):
    P, I32, I64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sig = {
        "dion_abi_version": (I32, []),
        "dion_status_string": (ctypes.c_char_p, [I32]),
        "dion_last_error": (ctypes.c_char_p, []),
        "dion_plan_create": (I32, [ctypes.POINTER(MatrixDesc), I32, ctypes.POINTER(SZ), ctypes.POINTER(P)]),
        "dion_plan_destroy": (None, [P]),
        "dion_plan_count": (I32, [P]),
        "dion_plan_set_hparams": (I32, [P, I32, F, F]),
        "dion_plan_upload": (I32, [P, P, SZ, P]),
        "dion_step_batched": (I32, [P, P, SZ, P]),
        "dion_step_phases": (I32, [P, P, SZ, I32, I32, P]),
        "dion_plan_buffer": (I32, [P, I32, I32, ctypes.POINTER(SZ), ctypes.POINTER(I64),
                                   ctypes.POINTER(I64), ctypes.POINTER(I64)]),
        "dion_plan_get_status": (I32, [P, P, SZ, ctypes.POINTER(ctypes.c_uint32), P]),
        "dion_plan_launches_per_step": (I32, [P]),
        "dion_orth_noalloc": (I32, [P, I64, I64, I64, P, I64, ctypes.POINTER(ctypes.c_uint32), P]),
        "dion_debug_expire_wait": (I32, [I64, I32, P]),
        "dion_shard_stage": (I32, [P, P, SZ, I32, P]),
        "dion_plan_exchange": (I32, [P, I32, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]),
        "muon_plan_create": (I32, [ctypes.POINTER(MuonDesc), I32, I32, I32, F, ctypes.POINTER(SZ),
                                   ctypes.POINTER(P)]),
        "muon_plan_selected_rows": (I32, [P, I32, ctypes.POINTER(SZ), ctypes.POINTER(I64)]),
        "muon_step_batched": (I32, [P, P, SZ, P]),
        "muon_plan_launches_per_step": (I32, [P]),
        "muon_plan_destroy": (None, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """The loaded libdion.so (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdion.so is not built ({LIB_PATH}); run "
                               "python -m rank_orthonormalized_optimizer_03_b300.build")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def header_functions() -> List[str]:
    """Names of the functions declared in the headers under include/."""
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if h.endswith(".h"):
            txt = open(os.path.join(INCLUDE, h)).read()
            names |= set(re.findall(r"DION_API\s+[\w\s\*]+?\b((?:dion|muon)_\w+)\s*\(", txt))
    return sorted(names)


def check(code: int, where: str):
    if code != DION_OK:
        raise DionError(code, where, lib().dion_last_error().decode())


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return int(getattr(stream, "cuda_stream", stream)) or None


def _check_device(tensors, names, device=None):
    """Every tensor a CUDA tensor on one device (the library takes device pointers)."""
    for t, nm in zip(tensors, names):
        if not t.is_cuda:
            raise ValueError(f"{nm} must be a CUDA tensor (got {t.device})")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError(f"{nm} is on {t.device}, expected {device}")
    return device


def make_desc(X, G, R, V, eta, beta, variant="orth", scale=0.0) -> MatrixDesc:
    """Descriptor for one matrix from torch tensors (row-major, unit column stride)."""
    import torch
    if X.dim() != 2:
        raise ValueError("X must be an m x n matrix")
    m, n = X.shape
    r = V.shape[1]
    for t, nm in ((X, "X"), (G, "G"), (R, "R")):
        if t.dim() != 2 or t.shape != (m, n) or t.stride(1) != 1:
            raise ValueError(f"{nm} must be an m x n row-major view")
    if X.dtype != torch.float32 or R.dtype != torch.float32 or V.dtype != torch.float32:
        raise ValueError("X, R, V must be float32")
    if G.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("G must be float32 or bfloat16")
    if V.dim() != 2 or V.shape != (n, r) or not V.is_contiguous():
        raise ValueError("V must be a contiguous n x r tensor")
    if variant not in VARIANT:
        raise ValueError(f"variant must be one of {sorted(VARIANT)}")
    _check_device((X, G, R, V), ("X", "G", "R", "V"))
    return MatrixDesc(
        X.data_ptr(), G.data_ptr(), R.data_ptr(), V.data_ptr(), m, n, r,
        X.stride(0), G.stride(0), R.stride(0),
        DTYPE_BF16 if G.dtype == torch.bfloat16 else DTYPE_F32, VARIANT[variant],
        float(eta), float(beta), float(scale), 0.0)


def debug_expire_wait(limit_ns: int = 0, withhold_matrix: int = -1, stream=None):
    """Testing hook of the bounded waits (dion_debug_expire_wait): wait limit in ns
    (<= 0: the 2 s default) and the plan matrix whose update operands the update
    kernel withholds (-1: none).  Process-wide; reset with debug_expire_wait()."""
    check(lib().dion_debug_expire_wait(int(limit_ns), int(withhold_matrix), _stream_ptr(stream)),
          "dion_debug_expire_wait")


NOALLOC_MAX_ROWS, NOALLOC_MAX_RANK = 8192, 64


def orth_noalloc(A, Q, stream=None, status: bool = True) -> Optional[int]:
    """Q = orth(A) for one matrix through dion_orth_noalloc (no device allocation
    in the library; its scratch is a fixed array inside libdion.so).

    A and Q are float32 CUDA tensors (rows x r views with unit column stride).
    With status=True the call waits for the result and returns the matrix's
    status word; otherwise it returns None without waiting.  Inside a stream
    capture pass status=False (the status copy and the wait are not allowed
    there).
    """
    import torch
    if A.dim() != 2 or Q.dim() != 2 or A.shape != Q.shape:
        raise ValueError("A and Q must be rows x r matrices of the same shape")
    if A.dtype != torch.float32 or Q.dtype != torch.float32 or A.stride(1) != 1 or Q.stride(1) != 1:
        raise ValueError("A and Q must be float32 with unit column stride")
    _check_device((A, Q), ("A", "Q"))
    if status and torch.cuda.is_current_stream_capturing():
        raise RuntimeError("orth_noalloc: pass status=False while the stream is being captured")
    rows, r = A.shape
    st = ctypes.c_uint32(0)
    check(lib().dion_orth_noalloc(A.data_ptr(), rows, r, A.stride(0), Q.data_ptr(), Q.stride(0),
                                  ctypes.byref(st) if status else None, _stream_ptr(stream)), "dion_orth_noalloc")
    return st.value if status else None


class Plan:
    """A batch of matrices stepped together (one grouped launch per phase).

    ``mats`` is a sequence of dicts with keys X, G, R, V (CUDA tensors owned by
    the caller and updated in place) and eta, beta, variant ("orth" | "dion" |
    "lowrank_muon"; with "lowrank_muon" R holds Muon's momentum, beta is its
    coefficient and V must hold a fresh sketch before every step), optional
    scale (<= 0 or missing: sqrt(m/n)).  The workspace is a torch
    uint8 tensor allocated here unless one is passed in.
    """

    def __init__(self, mats: Sequence[dict], workspace=None, device=None):
        import torch
        L = lib()
        if len(mats) == 0:
            raise ValueError("a plan needs at least one matrix")
        dev0 = mats[0]["X"].device
        for k, d in enumerate(mats):
            for key in ("X", "G", "R", "V"):
                if d[key].device != dev0:
                    raise ValueError(f"matrix {k}: {key} is on {d[key].device}, the plan's first X on {dev0}")
        self._keep = [(d["X"], d["G"], d["R"], d["V"]) for d in mats]
        descs = (MatrixDesc * len(mats))(*[
            make_desc(d["X"], d["G"], d["R"], d["V"], d["eta"], d["beta"], d.get("variant", "orth"),
                      d.get("scale", 0.0)) for d in mats])
        self._descs = descs
        ws = ctypes.c_size_t(0)
        plan = ctypes.c_void_p()
        check(L.dion_plan_create(descs, len(mats), ctypes.byref(ws), ctypes.byref(plan)), "dion_plan_create")
        self._plan = plan
        self.count = len(mats)
        self.ws_bytes = ws.value
        if workspace is None:
            dev = device if device is not None else mats[0]["X"].device
            workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        if workspace.dtype != torch.uint8 or workspace.dim() != 1:
            raise ValueError("workspace must be a 1-D uint8 tensor")
        if workspace.numel() < self.ws_bytes:
            raise ValueError("workspace too small")
        if workspace.device != mats[0]["X"].device:
            raise ValueError("workspace must be on the matrices' device")
        self.workspace = workspace

    def close(self):
        if getattr(self, "_plan", None):
            lib().dion_plan_destroy(self._plan)
            self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def launches_per_step(self) -> int:
        return lib().dion_plan_launches_per_step(self._plan)

    def upload(self, stream=None):
        check(lib().dion_plan_upload(self._plan, self.workspace.data_ptr(), self.ws_bytes,
                                     _stream_ptr(stream)), "dion_plan_upload")

    def step(self, stream=None):
        check(lib().dion_step_batched(self._plan, self.workspace.data_ptr(), self.ws_bytes,
                                      _stream_ptr(stream)), "dion_step_batched")

    def phases(self, first: int, last: int, stream=None):
        check(lib().dion_step_phases(self._plan, self.workspace.data_ptr(), self.ws_bytes, first, last,
                                     _stream_ptr(stream)), "dion_step_phases")

    def set_hparams(self, idx: int, eta: float, beta: float):
        check(lib().dion_plan_set_hparams(self._plan, idx, eta, beta), "dion_plan_set_hparams")

    def failures(self, stream=None) -> List[int]:
        """Per-matrix status words restricted to the bits that mean "not updated"."""
        return [v & FATAL for v in self.status(stream)]

    def status(self, stream=None) -> List[int]:
        out = (ctypes.c_uint32 * self.count)()
        check(lib().dion_plan_get_status(self._plan, self.workspace.data_ptr(), self.ws_bytes, out,
                                         _stream_ptr(stream)), "dion_plan_get_status")
        return list(out)

    def buffer(self, idx: int, which: int):
        """A float32 view (rows x r) of intermediate P, U or W of matrix idx."""
        import torch
        off, rows, cols, ld = ctypes.c_size_t(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(lib().dion_plan_buffer(self._plan, idx, which, ctypes.byref(off), ctypes.byref(rows),
                                     ctypes.byref(cols), ctypes.byref(ld)), "dion_plan_buffer")
        nbytes = rows.value * ld.value * 4
        raw = self.workspace[off.value: off.value + nbytes]
        return raw.view(torch.float32).view(rows.value, ld.value)[:, : cols.value]


class MuonPlan:
    """The Muon comparator (include/muon.h) over a batch of matrices.

    ``mats`` is a sequence of dicts with keys X, G, B (CUDA tensors owned by the
    caller; X and the momentum B are float32 and updated in place, G float32 or
    bfloat16) and eta, mu, optional scale (<= 0 or missing: sqrt(m/n)).
    ``iters`` Newton-Schulz iterations in ``precision`` "bf16" | "tf32" | "fp32".
    ``row_fraction`` < 1 selects the Dion3 row-selection variant (only the
    ceil(row_fraction m) rows of largest norm are orthogonalised and updated).
    """

    def __init__(self, mats: Sequence[dict], iters: int = 5, precision: str = "bf16", workspace=None,
                 row_fraction: float = 1.0):
        import torch
        L = lib()
        if len(mats) == 0:
            raise ValueError("a plan needs at least one matrix")
        if precision not in MUON_PRECISION:
            raise ValueError(f"precision must be one of {sorted(MUON_PRECISION)}")
        descs = []
        dev0 = mats[0]["X"].device
        for k, d in enumerate(mats):
            X, G, B = d["X"], d["G"], d["B"]
            _check_device((X, G, B), ("X", "G", "B"), dev0)
            if X.dim() != 2 or G.shape != X.shape or B.shape != X.shape:
                raise ValueError(f"matrix {k}: X, G, B must be m x n matrices of one shape")
            if X.stride(1) != 1 or G.stride(1) != 1 or B.stride(1) != 1:
                raise ValueError(f"matrix {k}: X, G, B must be row-major views")
            if X.dtype != torch.float32 or B.dtype != torch.float32 or G.dtype not in (torch.float32, torch.bfloat16):
                raise ValueError(f"matrix {k}: X, B float32 and G float32 or bfloat16")
            m, n = X.shape
            descs.append(MuonDesc(X.data_ptr(), G.data_ptr(), B.data_ptr(), m, n, X.stride(0), G.stride(0),
                                  B.stride(0), DTYPE_BF16 if G.dtype == torch.bfloat16 else DTYPE_F32,
                                  float(d["eta"]), float(d["mu"]), float(d.get("scale", 0.0))))
        self._keep = [(d["X"], d["G"], d["B"]) for d in mats]
        self._descs = (MuonDesc * len(descs))(*descs)
        ws = ctypes.c_size_t(0)
        plan = ctypes.c_void_p()
        check(L.muon_plan_create(self._descs, len(descs), int(iters), MUON_PRECISION[precision],
                                 float(row_fraction), ctypes.byref(ws), ctypes.byref(plan)), "muon_plan_create")
        self._plan = plan
        self.ws_bytes = ws.value
        if workspace is None:
            workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev0)
        if workspace.dtype != torch.uint8 or workspace.dim() != 1 or workspace.numel() < self.ws_bytes:
            raise ValueError("workspace must be a 1-D uint8 tensor of at least ws_bytes")
        self.workspace = workspace

    @property
    def launches_per_step(self) -> int:
        return lib().muon_plan_launches_per_step(self._plan)

    def selected_rows(self, idx: int):
        """int32 view of the rows of matrix idx that the last step selected (row-selection variant)."""
        import torch
        off, k = ctypes.c_size_t(), ctypes.c_int64()
        check(lib().muon_plan_selected_rows(self._plan, idx, ctypes.byref(off), ctypes.byref(k)),
              "muon_plan_selected_rows")
        return self.workspace[off.value: off.value + 4 * k.value].view(torch.int32)

    def step(self, stream=None):
        check(lib().muon_step_batched(self._plan, self.workspace.data_ptr(), self.ws_bytes, _stream_ptr(stream)),
              "muon_step_batched")

    def close(self):
        if getattr(self, "_plan", None):
            lib().muon_plan_destroy(self._plan)
            self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def group_bounds(nbytes: Sequence[int], groups: int) -> List[tuple]:
    """Split items 0..len-1 into at most ``groups`` consecutive ranges of about
    equal total bytes (every range non-empty)."""
    groups = max(1, min(groups, len(nbytes)))
    total = float(sum(nbytes))
    cuts, acc = [0], 0.0
    for i, b in enumerate(nbytes[:-1]):
        acc += b
        # close a range once it reaches its share, leaving one item per remaining range
        if len(cuts) < groups and acc >= total * len(cuts) / groups and len(nbytes) - (i + 1) >= groups - len(cuts):
            cuts.append(i + 1)
    cuts.append(len(nbytes))
    return list(zip(cuts[:-1], cuts[1:]))


class HostFedStep:
    """Steps of a batch whose gradients arrive from pinned host memory.

    The matrices are split into ``groups`` consecutive groups of about equal
    gradient bytes, each with its own :class:`Plan`.  A group's gradients lie
    back to back (256-byte aligned) in one device slab and in one pinned host
    slab of the same layout: the caller writes matrix i's gradient into
    :meth:`host_grad` (i), and every step copies each group's host slab to its
    device slab in one transfer on a side stream, then steps the group on the
    caller's stream once the copy is in, so that the copy of group g + 1
    overlaps the step of group g.  A group's copy waits until the previous step
    of that group has read its gradients.  Matrix i's ``G`` in ``self.mats``
    is its view of the device slab (the caller's original G is copied in once
    and no longer read).  Each matrix gets the arithmetic of a plan over the
    whole batch whenever each group still fills the GPU (the K split of
    W = M^T U is the only choice that depends on the batch).
    """

    ALIGN = 256

    def __init__(self, mats: Sequence[dict], groups: int = 8):
        import torch
        self.mats = [dict(d) for d in mats]
        sizes = [d["G"].numel() * d["G"].element_size() for d in self.mats]
        self.ranges = group_bounds(sizes, groups)
        dev = self.mats[0]["X"].device
        self.dev_slabs, self.host_slabs, self._host_views = [], [], [None] * len(self.mats)
        for a, b in self.ranges:
            offs, tot = [], 0
            for i in range(a, b):
                offs.append(tot)
                tot += -(-sizes[i] // self.ALIGN) * self.ALIGN
            dslab = torch.empty(tot, dtype=torch.uint8, device=dev)
            hslab = torch.empty(tot, dtype=torch.uint8, pin_memory=True)
            for k, i in enumerate(range(a, b)):
                G = self.mats[i]["G"]
                dv = dslab[offs[k]: offs[k] + sizes[i]].view(G.dtype).view(G.shape)
                dv.copy_(G)
                self.mats[i]["G"] = dv
                self._host_views[i] = hslab[offs[k]: offs[k] + sizes[i]].view(G.dtype).view(G.shape)
            self.dev_slabs.append(dslab)
            self.host_slabs.append(hslab)
        self.plans = [Plan(self.mats[a:b]) for a, b in self.ranges]
        self.copy_stream = torch.cuda.Stream(device=dev)
        self._read = [None] * len(self.plans)   # per group: event after its last step

    def host_grad(self, i: int):
        """The pinned host buffer (a tensor view) that matrix i's gradient is read from.

        The copies are asynchronous: rewrite it for the next step only once the
        previous step's copy has completed (after :meth:`status`, or a
        synchronize of the stream passed to :meth:`step`)."""
        return self._host_views[i]

    def h2d_bytes(self) -> int:
        """Bytes copied host -> device per step (the group slabs, alignment padding included)."""
        return sum(h.numel() for h in self.host_slabs)

    def step(self, stream=None):
        """Copy every group's gradients in and step every group (asynchronous)."""
        import torch
        cs = stream if stream is not None else torch.cuda.current_stream()
        for g, (plan, dslab, hslab) in enumerate(zip(self.plans, self.dev_slabs, self.host_slabs)):
            ready = torch.cuda.Event()
            with torch.cuda.stream(self.copy_stream):
                if self._read[g] is not None:
                    self.copy_stream.wait_event(self._read[g])
                dslab.copy_(hslab, non_blocking=True)
                ready.record(self.copy_stream)
            cs.wait_event(ready)
            plan.step(cs)
            done = torch.cuda.Event()
            done.record(cs)
            self._read[g] = done

    def status(self, stream=None) -> List[int]:
        """Per-matrix status words of the last step, in batch order (synchronises)."""
        out: List[int] = []
        for p in self.plans:
            out += p.status(stream)
        return out

    def close(self):
        for p in self.plans:
            p.close()
