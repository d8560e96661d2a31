"""Thin ctypes binding of libjetscore (argument marshalling only).

Every step of the scoring head runs in the library's CUDA kernels; this module
only passes torch tensors' device pointers, sizes and the current CUDA stream
through the C ABI declared in ``include/jetscore.h``.  It has no CPU path: if
the library is not built, loading it raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional, Sequence

import torch

from . import build as _build

JET_OK = 0
JET_ERR_ARG = -1
JET_ERR_TOKEN_RANGE = -2
JET_ERR_OFFSETS = -3
JET_ERR_MODE = -4
JET_ERR_NOT_IN_UNION = -5
JET_ERR_WORKSPACE = -6
JET_ERR_UNSUPPORTED = -7
JET_ERR_CUDA = -8
JET_ERR_TIMEOUT = -9

JET_KIND_CHOICE, JET_KIND_BINARY, JET_KIND_ORDINAL = 0, 1, 2
JET_MODE_FULL, JET_MODE_RESTRICTED = 0, 1
JET_W_ROWMAJOR, JET_W_TILED = 0, 1
JET_MAX_UNION = 4096

SET_OUTPUTS = ("logp", "lse", "s", "q", "q_equiv", "decision", "expected", "confidence", "mass")


class JetError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class _SetOut(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in SET_OUTPUTS]


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> C.CDLL:
    """Load the in-tree libjetscore.so; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libjetscore is not built ({path} missing); run "
                           "candidate_answer_scoring_gb300.build.build() with the CUDA toolkit")
    lib = C.CDLL(path)
    P, I, F = C.c_void_p, C.c_int, C.c_float
    lib.jet_create.argtypes = [C.POINTER(P), I, I, I, I, I]
    lib.jet_destroy.argtypes = [P]
    lib.jet_destroy.restype = None
    lib.jet_status_string.argtypes = [I]
    lib.jet_status_string.restype = C.c_char_p
    lib.jet_score_tokens.argtypes = [P, P, P, P, I, P, P, P]
    sets_sig = [P, P, P, I, P, P, I, P, I, P, P, I, F, I, P, I, C.POINTER(_SetOut), P]
    for name in ("jet_score_sets", "jet_score_sets_async", "jet_score_sets_host", "jet_score_sets_host_async"):
        getattr(lib, name).argtypes = sets_sig
    lib.jet_host_wait.argtypes = [P, P]
    lib.jet_tiled_weights_bytes.argtypes = [P]
    lib.jet_tiled_weights_bytes.restype = C.c_size_t
    lib.jet_tile_weights.argtypes = [P, P, P, P]
    lib.jet_set_weights_layout.argtypes = [P, I]
    for name in ("jet_score_sets_gather", "jet_score_sets_gather_async"):
        getattr(lib, name).argtypes = [P, P, I, P, I, P, P, P, I, P, I, P, P, I, F, I, P, I, C.POINTER(_SetOut), P]
    lib.jet_sync_status.argtypes = [P, P]
    lib.jet_plan_info.argtypes = [P, I, C.POINTER(C.c_int)]
    lib.jet_profile_enable.argtypes = [P, I]
    lib.jet_profile_read.argtypes = [P, C.POINTER(C.c_double), I]
    lib.jet_selftest_wait_timeout.argtypes = [P, I, P]
    lib.jet_dedup_rows.argtypes = [P, P, I, P, I, P, P, P, C.POINTER(C.c_int), P]
    lib.jet_layer_sensitivity.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P]
    lib.jet_fit_temperature.argtypes = [P, P, P, I, P, I, P, I, P, C.c_double, C.c_double,
                                        C.POINTER(C.c_double), C.POINTER(C.c_double), P]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().jet_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_dev(t: torch.Tensor, name: str, device: torch.device, dtypes: Sequence[torch.dtype]):
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a tensor on {device}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)


class JetScorer:
    """A libjetscore context: output embedding shape [V, d] and a workspace for
    up to ``max_rows`` hidden rows and ``max_tokens`` scored tokens per call."""

    def __init__(self, d: int, V: int, max_rows: int, max_tokens: int, device: int = 0):
        self.lib = load()
        self.d, self.V, self.max_rows, self.max_tokens = d, V, max_rows, max_tokens
        self.device = torch.device("cuda", device)
        h = C.c_void_p()
        rc = self.lib.jet_create(C.byref(h), d, V, max_rows, max_tokens, device)
        if rc != JET_OK:
            raise JetError(rc, "jet_create")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None):
            self.lib.jet_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -------------------------------------------------------------- calls
    def plan_info(self, n_rows: int) -> Dict[str, int]:
        out = (C.c_int * 8)()
        rc = self.lib.jet_plan_info(self._h, int(n_rows), out)
        if rc != JET_OK:
            raise JetError(rc, "jet_plan_info")
        keys = ("row_tiles", "vocab_tiles", "splits", "band_height", "units", "ctas", "tile_rows", "tile_cols")
        return dict(zip(keys, list(out)))

    def score_tokens(self, H: torch.Tensor, W: torch.Tensor, tok_ids: torch.Tensor, want_lse: bool = False):
        """logp[i] = log softmax_V(H[i] W^T)[tok_ids[i]] (and lse[i])."""
        dev = self.device
        _check_dev(H, "H", dev, _BF16); _check_dev(W, "W", dev, _BF16)
        _check_dev(tok_ids, "tok_ids", dev, (torch.int32,))
        n = tok_ids.numel()
        logp = torch.empty(n, dtype=torch.float32, device=dev)
        lse = torch.empty(n, dtype=torch.float32, device=dev) if want_lse else None
        rc = self.lib.jet_score_tokens(self._h, _ptr(H), _ptr(W), _ptr(tok_ids), n, _ptr(logp), _ptr(lse),
                                       _stream(dev))
        if rc != JET_OK:
            raise JetError(rc, "jet_score_tokens")
        return (logp, lse) if want_lse else logp

    def alloc_outputs(self, n_rows: int, n_tok: int, n_cand: int, n_sets: int,
                      want: Sequence[str] = SET_OUTPUTS) -> Dict[str, torch.Tensor]:
        dev = self.device
        sizes = dict(logp=n_tok, lse=n_rows, s=n_cand, q=n_cand, q_equiv=n_cand, decision=n_sets,
                     expected=n_sets, confidence=n_sets, mass=n_sets)
        return {k: torch.empty(sizes[k], dtype=torch.int32 if k == "decision" else torch.float32, device=dev)
                for k in want}

    def _set_args(self, H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T, mode, union_ids, out):
        so = _SetOut(*[_ptr(out.get(n)) for n in SET_OUTPUTS])
        n_union = 0 if union_ids is None else union_ids.numel()
        args = [self._h, _ptr(H), _ptr(W), H.shape[0], _ptr(tok_row), _ptr(tok_ids), tok_ids.numel(),
                _ptr(cand_offsets), cand_offsets.numel() - 1, _ptr(set_offsets), _ptr(kind),
                set_offsets.numel() - 1, C.c_float(T), int(mode), _ptr(union_ids), n_union, C.byref(so)]
        return args, so

    def score_sets(self, H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float,
                   mode: int = JET_MODE_FULL, union_ids=None, out: Optional[Dict[str, torch.Tensor]] = None,
                   sync: bool = True) -> Dict[str, torch.Tensor]:
        """Whole scoring head on device tensors; returns the output tensors."""
        dev = self.device
        _check_dev(H, "H", dev, _BF16); _check_dev(W, "W", dev, _BF16)
        for name, t in (("tok_row", tok_row), ("tok_ids", tok_ids), ("cand_offsets", cand_offsets),
                        ("set_offsets", set_offsets)):
            _check_dev(t, name, dev, (torch.int32,))
        _check_dev(kind, "kind", dev, (torch.uint8,))
        if union_ids is not None:
            _check_dev(union_ids, "union_ids", dev, (torch.int32,))
        if out is None:
            out = self.alloc_outputs(H.shape[0], tok_ids.numel(), cand_offsets.numel() - 1,
                                     set_offsets.numel() - 1)
        args, keep = self._set_args(H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T, mode, union_ids,
                                    out)
        fn = self.lib.jet_score_sets if sync else self.lib.jet_score_sets_async
        rc = fn(*args, _stream(dev))
        if rc != JET_OK:
            raise JetError(rc, "jet_score_sets")
        return out

    def score_sets_gather(self, H_src, row_index, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float,
                          mode: int = JET_MODE_FULL, union_ids=None,
                          out: Optional[Dict[str, torch.Tensor]] = None, sync: bool = True) -> Dict[str, torch.Tensor]:
        """score_sets with row i of the problem read in place as H_src[row_index[i]]
        (e.g. the answer positions of a right-padded [B*L, d] backbone output)."""
        dev = self.device
        _check_dev(H_src, "H_src", dev, _BF16); _check_dev(W, "W", dev, _BF16)
        for name, t in (("row_index", row_index), ("tok_row", tok_row), ("tok_ids", tok_ids),
                        ("cand_offsets", cand_offsets), ("set_offsets", set_offsets)):
            _check_dev(t, name, dev, (torch.int32,))
        _check_dev(kind, "kind", dev, (torch.uint8,))
        if union_ids is not None:
            _check_dev(union_ids, "union_ids", dev, (torch.int32,))
        n_rows = row_index.numel()
        if out is None:
            out = self.alloc_outputs(n_rows, tok_ids.numel(), cand_offsets.numel() - 1, set_offsets.numel() - 1)
        so = _SetOut(*[_ptr(out.get(n)) for n in SET_OUTPUTS])
        n_union = 0 if union_ids is None else union_ids.numel()
        fn = self.lib.jet_score_sets_gather if sync else self.lib.jet_score_sets_gather_async
        rc = fn(
            self._h, _ptr(H_src), H_src.shape[0], _ptr(row_index), n_rows, _ptr(W), _ptr(tok_row), _ptr(tok_ids),
            tok_ids.numel(), _ptr(cand_offsets), cand_offsets.numel() - 1, _ptr(set_offsets), _ptr(kind),
            set_offsets.numel() - 1, C.c_float(T), int(mode), _ptr(union_ids), n_union, C.byref(so), _stream(dev))
        if rc != JET_OK:
            raise JetError(rc, "jet_score_sets_gather")
        return out

    def tile_weights(self, W: torch.Tensor, use: bool = True) -> torch.Tensor:
        """The tiled copy of W ([ceil(V/128)*128, d] bf16 in 16 KB boxes, rows
        past V zero) that the head streams fastest; with use=True the scorer's
        later calls read their W argument in this layout."""
        _check_dev(W, "W", self.device, _BF16)
        n = self.lib.jet_tiled_weights_bytes(self._h) // 2
        Wt = torch.empty(n // self.d, self.d, dtype=W.dtype, device=self.device)
        rc = self.lib.jet_tile_weights(self._h, _ptr(W), _ptr(Wt), _stream(self.device))
        if rc != JET_OK:
            raise JetError(rc, "jet_tile_weights")
        if use:
            self.set_weights_layout(JET_W_TILED)
        return Wt

    def set_weights_layout(self, layout: int) -> None:
        """How later calls read W: JET_W_ROWMAJOR (default) or JET_W_TILED."""
        rc = self.lib.jet_set_weights_layout(self._h, int(layout))
        if rc != JET_OK:
            raise JetError(rc, "jet_set_weights_layout")

    KERNELS = ("prep", "head", "merge", "restricted", "sets")

    def profile(self, enable: bool) -> None:
        rc = self.lib.jet_profile_enable(self._h, 1 if enable else 0)
        if rc != JET_OK:
            raise JetError(rc, "jet_profile_enable")

    def profile_read(self) -> Dict[str, Dict[str, float]]:
        """Per kernel kind: launches and total device milliseconds since the last read."""
        out = (C.c_double * 11)()
        rc = self.lib.jet_profile_read(self._h, out, 11)
        if rc != JET_OK:
            raise JetError(rc, "jet_profile_read")
        res = {k: {"launches": int(out[2 * i]), "ms": float(out[2 * i + 1])} for i, k in enumerate(self.KERNELS)}
        res["untimed_launches"] = int(out[10])
        return res

    def dedup_rows(self, H: torch.Tensor, tok_row: torch.Tensor, H_unique: Optional[torch.Tensor] = None,
                   want_row_map: bool = False):
        """Distinct rows of H (first occurrences, in order) and the tokens' rows
        in them: returns (H_unique[:n_unique], tok_row_unique, row_map or None)."""
        dev = self.device
        _check_dev(H, "H", dev, _BF16)
        _check_dev(tok_row, "tok_row", dev, (torch.int32,))
        if H_unique is None:
            H_unique = torch.empty_like(H)
        tok_u = torch.empty_like(tok_row)
        row_map = torch.empty(H.shape[0], dtype=torch.int32, device=dev) if want_row_map else None
        n = C.c_int(0)
        rc = self.lib.jet_dedup_rows(self._h, _ptr(H), H.shape[0], _ptr(tok_row), tok_row.numel(), _ptr(H_unique),
                                     _ptr(tok_u), _ptr(row_map), C.byref(n), _stream(dev))
        if rc != JET_OK:
            raise JetError(rc, "jet_dedup_rows")
        return H_unique[:n.value], tok_u, row_map

    def fit_temperature(self, s, tok_ids, cand_offsets, set_offsets, gold, T_min: float = 0.05,
                        T_max: float = 100.0):
        """Temperature minimising the mean gold NLL; returns (T, nll)."""
        dev = self.device
        _check_dev(s, "s", dev, (torch.float32,))
        for name, t in (("tok_ids", tok_ids), ("cand_offsets", cand_offsets), ("set_offsets", set_offsets),
                        ("gold", gold)):
            _check_dev(t, name, dev, (torch.int32,))
        T, nll = C.c_double(0), C.c_double(0)
        rc = self.lib.jet_fit_temperature(self._h, _ptr(s), _ptr(tok_ids), tok_ids.numel(), _ptr(cand_offsets),
                                          cand_offsets.numel() - 1, _ptr(set_offsets), set_offsets.numel() - 1,
                                          _ptr(gold), float(T_min), float(T_max), C.byref(T), C.byref(nll),
                                          _stream(dev))
        if rc != JET_OK:
            raise JetError(rc, "jet_fit_temperature")
        return T.value, nll.value

    def layer_sensitivity(self, z, z_skip, offsets, k: int):
        """(d [L, n], J [L], selected [k]) of the layer-sensitivity ranking."""
        dev = self.device
        _check_dev(z, "z", dev, (torch.float32,))
        _check_dev(z_skip, "z_skip", dev, (torch.float32,))
        _check_dev(offsets, "offsets", dev, (torch.int32,))
        L, n = z_skip.shape[0], offsets.numel() - 1
        d = torch.empty((L, n), dtype=torch.float32, device=dev)
        J = torch.empty(L, dtype=torch.float32, device=dev)
        sel = torch.empty(max(k, 1), dtype=torch.int32, device=dev)
        rc = self.lib.jet_layer_sensitivity(self._h, _ptr(z), _ptr(z_skip), _ptr(offsets), n, z.numel(), L, int(k),
                                            _ptr(d), _ptr(J), _ptr(sel), _stream(dev))
        if rc != JET_OK:
            raise JetError(rc, "jet_layer_sensitivity")
        return d, J, sel[:k]

    def bind_dedup_rows(self, H: torch.Tensor, tok_row: torch.Tensor, H_unique: torch.Tensor,
                        tok_row_unique: torch.Tensor, row_map: Optional[torch.Tensor] = None):
        """dedup_rows with its checks and argument marshalling done once: returns
        call, where call() makes only the (synchronous) jet_dedup_rows C call into
        the given buffers and returns n_unique.  The tensors must stay alive and
        unchanged in shape while call is used; their contents may change."""
        dev = self.device
        _check_dev(H, "H", dev, _BF16)
        _check_dev(H_unique, "H_unique", dev, _BF16)
        for name, t in (("tok_row", tok_row), ("tok_row_unique", tok_row_unique)):
            _check_dev(t, name, dev, (torch.int32,))
        if row_map is not None:
            _check_dev(row_map, "row_map", dev, (torch.int32,))
        if H_unique.shape != H.shape or tok_row_unique.numel() != tok_row.numel() or \
                (row_map is not None and row_map.numel() != H.shape[0]):
            raise ValueError("dedup_rows buffers do not match H and tok_row")
        n = C.c_int(0)
        args = (self._h, _ptr(H), H.shape[0], _ptr(tok_row), tok_row.numel(), _ptr(H_unique), _ptr(tok_row_unique),
                _ptr(row_map), C.byref(n), _stream(dev))
        fn = self.lib.jet_dedup_rows
        held = (H, tok_row, H_unique, tok_row_unique, row_map)

        def call():
            rc = fn(*args)
            if rc != JET_OK:
                raise JetError(rc, "jet_dedup_rows")
            return n.value

        call.buffers = held   # the marshalled pointers stay valid while call lives
        return call

    def bind_fit_temperature(self, s, tok_ids, cand_offsets, set_offsets, gold, T_min: float = 0.05,
                             T_max: float = 100.0):
        """fit_temperature marshalled once: returns call, where call() makes only
        the (synchronous) jet_fit_temperature C call and returns (T, nll)."""
        dev = self.device
        _check_dev(s, "s", dev, (torch.float32,))
        for name, t in (("tok_ids", tok_ids), ("cand_offsets", cand_offsets), ("set_offsets", set_offsets),
                        ("gold", gold)):
            _check_dev(t, name, dev, (torch.int32,))
        T, nll = C.c_double(0), C.c_double(0)
        args = (self._h, _ptr(s), _ptr(tok_ids), tok_ids.numel(), _ptr(cand_offsets), cand_offsets.numel() - 1,
                _ptr(set_offsets), set_offsets.numel() - 1, _ptr(gold), float(T_min), float(T_max), C.byref(T),
                C.byref(nll), _stream(dev))
        fn = self.lib.jet_fit_temperature
        held = (s, tok_ids, cand_offsets, set_offsets, gold)

        def call():
            rc = fn(*args)
            if rc != JET_OK:
                raise JetError(rc, "jet_fit_temperature")
            return T.value, nll.value

        call.buffers = held
        return call

    def bind_layer_sensitivity(self, z, z_skip, offsets, k: int, d: torch.Tensor, J: torch.Tensor,
                               selected: torch.Tensor):
        """layer_sensitivity marshalled once, writing into d [L, n], J [L] and
        selected [k]: returns call, where call() makes only the (synchronous)
        jet_layer_sensitivity C call."""
        dev = self.device
        for name, t in (("z", z), ("z_skip", z_skip), ("d", d), ("J", J)):
            _check_dev(t, name, dev, (torch.float32,))
        for name, t in (("offsets", offsets), ("selected", selected)):
            _check_dev(t, name, dev, (torch.int32,))
        L, n = z_skip.shape[0], offsets.numel() - 1
        if d.numel() != L * n or J.numel() != L or selected.numel() < max(int(k), 1):
            raise ValueError("layer_sensitivity buffers do not match z_skip, offsets and k")
        args = (self._h, _ptr(z), _ptr(z_skip), _ptr(offsets), n, z.numel(), L, int(k), _ptr(d), _ptr(J),
                _ptr(selected), _stream(dev))
        fn = self.lib.jet_layer_sensitivity
        held = (z, z_skip, offsets, d, J, selected)

        def call():
            rc = fn(*args)
            if rc != JET_OK:
                raise JetError(rc, "jet_layer_sensitivity")

        call.buffers = held
        return call

    def selftest_wait_timeout(self, limit_us: int) -> int:
        """Run the bounded-wait diagnostic; returns the status (JET_ERR_TIMEOUT expected)."""
        return self.lib.jet_selftest_wait_timeout(self._h, int(limit_us), _stream(self.device))

    def sync_status(self) -> int:
        return self.lib.jet_sync_status(self._h, _stream(self.device))

    def score_sets_host(self, H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float,
                        mode: int = JET_MODE_FULL, union_ids=None,
                        out: Optional[Dict[str, torch.Tensor]] = None) -> Dict[str, torch.Tensor]:
        """End-to-end call with HOST (CPU, ideally pinned) tensors; W stays on the device."""
        _check_dev(W, "W", self.device, _BF16)
        cpu = torch.device("cpu")
        _check_dev(H, "H", cpu, _BF16)
        for name, t in (("tok_row", tok_row), ("tok_ids", tok_ids), ("cand_offsets", cand_offsets),
                        ("set_offsets", set_offsets)):
            _check_dev(t, name, cpu, (torch.int32,))
        _check_dev(kind, "kind", cpu, (torch.uint8,))
        if out is None:
            n = (H.shape[0], tok_ids.numel(), cand_offsets.numel() - 1, set_offsets.numel() - 1)
            sizes = dict(logp=n[1], lse=n[0], s=n[2], q=n[2], q_equiv=n[2], decision=n[3], expected=n[3],
                         confidence=n[3], mass=n[3])
            out = {k: torch.empty(v, dtype=torch.int32 if k == "decision" else torch.float32).pin_memory()
                   for k, v in sizes.items()}
        args, keep = self._set_args(H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T, mode, union_ids,
                                    out)
        rc = self.lib.jet_score_sets_host(*args, _stream(self.device))
        if rc != JET_OK:
            raise JetError(rc, "jet_score_sets_host")
        return out

    def bind_call(self, H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float,
                  mode: int = JET_MODE_FULL, union_ids=None, out: Optional[Dict[str, torch.Tensor]] = None,
                  sync: bool = False):
        """score_sets on device tensors with its checks and argument marshalling
        done once: returns (call, out), where call() makes only the
        jet_score_sets_async C call (jet_score_sets with sync=True) on the
        stream current at bind time, as a C caller holding these buffers would,
        and raises JetError on a non-zero status.  The tensors must stay alive
        and unchanged in shape while call is used; their contents may change
        between calls."""
        dev = self.device
        _check_dev(H, "H", dev, _BF16); _check_dev(W, "W", dev, _BF16)
        for name, t in (("tok_row", tok_row), ("tok_ids", tok_ids), ("cand_offsets", cand_offsets),
                        ("set_offsets", set_offsets)):
            _check_dev(t, name, dev, (torch.int32,))
        _check_dev(kind, "kind", dev, (torch.uint8,))
        if union_ids is not None:
            _check_dev(union_ids, "union_ids", dev, (torch.int32,))
        if out is None:
            out = self.alloc_outputs(H.shape[0], tok_ids.numel(), cand_offsets.numel() - 1,
                                     set_offsets.numel() - 1)
        args, keep = self._set_args(H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T, mode, union_ids,
                                    out)
        args = tuple(args) + (_stream(dev),)
        fn = self.lib.jet_score_sets if sync else self.lib.jet_score_sets_async
        held = (H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, union_ids, out, keep)

        def call():
            rc = fn(*args)
            if rc != JET_OK:
                raise JetError(rc, "jet_score_sets")
            return held

        return call, out

    def bind_gather_call(self, H_src, row_index, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float,
                         mode: int = JET_MODE_FULL, union_ids=None, out: Optional[Dict[str, torch.Tensor]] = None):
        """score_sets_gather marshalled once: returns (call, out), where call()
        makes only the jet_score_sets_gather_async C call on the stream current
        at bind time (the same contract as bind_call)."""
        dev = self.device
        _check_dev(H_src, "H_src", dev, _BF16); _check_dev(W, "W", dev, _BF16)
        for name, t in (("row_index", row_index), ("tok_row", tok_row), ("tok_ids", tok_ids),
                        ("cand_offsets", cand_offsets), ("set_offsets", set_offsets)):
            _check_dev(t, name, dev, (torch.int32,))
        _check_dev(kind, "kind", dev, (torch.uint8,))
        if union_ids is not None:
            _check_dev(union_ids, "union_ids", dev, (torch.int32,))
        n_rows = row_index.numel()
        if out is None:
            out = self.alloc_outputs(n_rows, tok_ids.numel(), cand_offsets.numel() - 1, set_offsets.numel() - 1)
        so = _SetOut(*[_ptr(out.get(n)) for n in SET_OUTPUTS])
        n_union = 0 if union_ids is None else union_ids.numel()
        args = (self._h, _ptr(H_src), H_src.shape[0], _ptr(row_index), n_rows, _ptr(W), _ptr(tok_row),
                _ptr(tok_ids), tok_ids.numel(), _ptr(cand_offsets), cand_offsets.numel() - 1, _ptr(set_offsets),
                _ptr(kind), set_offsets.numel() - 1, C.c_float(T), int(mode), _ptr(union_ids), n_union,
                C.byref(so), _stream(dev))
        fn = self.lib.jet_score_sets_gather_async
        held = (H_src, row_index, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, union_ids, out, so)

        def call():
            rc = fn(*args)
            if rc != JET_OK:
                raise JetError(rc, "jet_score_sets_gather")
            return held

        return call, out

    def bind_host_call(self, H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T: float,
                       mode: int = JET_MODE_FULL, union_ids=None,
                       out: Optional[Dict[str, torch.Tensor]] = None, pipelined: bool = False):
        """score_sets_host with its checks and argument marshalling done once:
        returns (call, out), where call() makes only the jet_score_sets_host
        C call on the current stream (as a C caller holding these buffers
        would) and raises JetError on a non-zero status.  The tensors must stay
        alive and unchanged in shape while call is used; their contents may
        change between calls.  With pipelined=True the call is
        jet_score_sets_host_async: it returns after enqueueing (the host
        tensors must be pinned), consecutive calls overlap their input copies
        with the previous call's kernels, and host_wait() collects them."""
        _check_dev(W, "W", self.device, _BF16)
        cpu = torch.device("cpu")
        _check_dev(H, "H", cpu, _BF16)
        for name, t in (("tok_row", tok_row), ("tok_ids", tok_ids), ("cand_offsets", cand_offsets),
                        ("set_offsets", set_offsets)):
            _check_dev(t, name, cpu, (torch.int32,))
        _check_dev(kind, "kind", cpu, (torch.uint8,))
        if union_ids is not None:
            _check_dev(union_ids, "union_ids", cpu, (torch.int32,))
        if out is None:
            n = (H.shape[0], tok_ids.numel(), cand_offsets.numel() - 1, set_offsets.numel() - 1)
            sizes = dict(logp=n[1], lse=n[0], s=n[2], q=n[2], q_equiv=n[2], decision=n[3], expected=n[3],
                         confidence=n[3], mass=n[3])
            out = {k: torch.empty(v, dtype=torch.int32 if k == "decision" else torch.float32).pin_memory()
                   for k, v in sizes.items()}
        args, keep = self._set_args(H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, T, mode, union_ids,
                                    out)
        args = tuple(args) + (_stream(self.device),)
        fn = self.lib.jet_score_sets_host_async if pipelined else self.lib.jet_score_sets_host
        held = (H, W, tok_row, tok_ids, cand_offsets, set_offsets, kind, union_ids, out, keep)

        def call():
            rc = fn(*args)
            if rc != JET_OK:
                raise JetError(rc, "jet_score_sets_host")
            return held

        return call, out

    def host_wait(self) -> int:
        """Wait for the pipelined host calls (bind_host_call(pipelined=True))
        enqueued since the last wait on the current stream; returns the first
        non-zero device status among them (0 if none)."""
        return int(self.lib.jet_host_wait(self._h, _stream(self.device)))
