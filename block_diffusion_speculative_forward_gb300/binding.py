"""Thin ctypes binding of libdflash (include/dflash.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, status codes become exceptions. Every step of
the draft head runs in the library's CUDA kernels. Loading fails loudly when
the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdflash.so")

OK, DECLINED, BOOKKEEPING_ONLY = 0, 1, 2
ERRORS = {-1: "EINVAL", -2: "ENOMEM", -3: "ESTATE", -4: "EPOSITION", -5: "ECUDA", -6: "EDEVICE"}
LAYER_KEYS = ("in_norm", "q", "k", "v", "q_norm", "k_norm", "o", "post_norm", "gate", "up", "down")


class DFlashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = ERRORS.get(code, str(code))


class Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("num_layers", "hidden", "intermediate", "num_q_heads",
                                          "num_kv_heads", "head_dim", "vocab", "gamma")] + [
        ("mask_token_id", C.c_uint32), ("n_target_layers", C.c_int32),
        ("target_hidden", C.c_int32), ("fc_in_features", C.c_int32), ("rms_eps", C.c_float),
        ("ctx_window", C.c_int32), ("kv_block", C.c_int32), ("prefill_chunk", C.c_int32),
        ("max_batch", C.c_int32), ("max_seq_len", C.c_int32), ("kv_pool_blocks", C.c_int32),
        ("kv_dtype", C.c_int32), ("lm_head_dtype", C.c_int32), ("rope_attn_factor", C.c_float),
        ("shifted_rows", C.c_int32)]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("lm_head_fp8", C.c_void_p),
                ("lm_head_scale", C.c_void_p), ("fc", C.c_void_p), ("hidden_norm", C.c_void_p),
                ("norm", C.c_void_p), ("inv_freq", C.c_void_p), ("kv_scale", C.c_void_p),
                ("layers", C.POINTER(C.c_void_p)), ("lm_head_nvfp4", C.c_void_p),
                ("lm_head_nvfp4_scale", C.c_void_p), ("lm_head_nvfp4_global", C.c_float)]


_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it is missing (no fallback exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libdflash.so is not built ({_LIB_PATH}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(_LIB_PATH)
        vp, i32, i64, u32 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint32
        sig = {
            "dflash_create": (C.c_int, [C.POINTER(Config), C.POINTER(Weights), C.POINTER(vp)]),
            "dflash_destroy": (None, [vp]),
            "dflash_propose_batch_max": (C.c_int, [vp]),
            "dflash_block_gamma": (C.c_int, [vp]),
            "dflash_alloc_state": (C.c_int, [vp, i64, C.POINTER(vp)]),
            "dflash_free_state": (C.c_int, [vp, vp]),
            "dflash_prefill": (C.c_int, [vp, vp, vp, i32, vp]),
            "dflash_propose": (C.c_int, [vp, vp, u32, i64, vp, i32, i32, vp, C.POINTER(u32),
                                         C.POINTER(i32), C.POINTER(C.c_float), vp]),
            "dflash_propose_batch": (C.c_int, [vp, i32, C.POINTER(vp), C.POINTER(u32),
                                               C.POINTER(i64), C.POINTER(vp), C.POINTER(i32), i32,
                                               vp, C.POINTER(u32), C.POINTER(i32),
                                               C.POINTER(C.c_float), vp]),
            "dflash_after_verify": (C.c_int, [vp, vp, i32]),
            "dflash_after_verify_batch": (C.c_int, [vp, i32, C.POINTER(vp), C.POINTER(i32)]),
            "dflash_catchup_batch": (C.c_int, [vp, i32, C.POINTER(vp), C.POINTER(vp),
                                               C.POINTER(vp), C.POINTER(i32), C.POINTER(i64),
                                               C.POINTER(i64), vp]),
            "dflash_take_drafter_kv": (C.c_int, [vp, vp, C.POINTER(i32), i32, C.POINTER(i32),
                                                 C.POINTER(i64)]),
            "dflash_install_drafter_kv": (C.c_int, [vp, vp, C.POINTER(i32), i32, i64]),
            "dflash_free_drafter_kv": (C.c_int, [vp, C.POINTER(i32), i32]),
            "dflash_yarn_inv_freq": (C.c_int, [C.c_double, i32, C.c_double, C.c_double,
                                               C.c_double, i32, C.POINTER(C.c_float),
                                               C.POINTER(C.c_float)]),
            "dflash_last_error": (C.c_char_p, []),
            "dflash_debug_state": (C.c_int, [vp, C.POINTER(i64), C.POINTER(i32), C.POINTER(i32), i32]),
            "dflash_debug_pool": (C.c_int, [vp, C.POINTER(i32), C.POINTER(i32)]),
            "dflash_debug_gather_kv": (C.c_int, [vp, vp, i32, i64, i32, vp, vp, vp]),
            "dflash_debug_set_taps": (C.c_int, [vp, vp, vp, vp]),
            "dflash_debug_set_graphs": (C.c_int, [vp, i32]),
            "dflash_debug_set_fault": (C.c_int, [vp, i64]),
            "dflash_debug_set_chain": (C.c_int, [vp, i32]),
            "dflash_debug_last_path": (C.c_int, [vp]),
            "dflash_debug_rows": (C.c_int, [vp, i32, C.POINTER(i32), C.POINTER(C.c_float), vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(rc: int, allow=(OK,)) -> int:
    if rc in allow:
        return rc
    raise DFlashError(rc, lib().dflash_last_error().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


_HAS_CUDA = None


def _stream() -> int | None:
    global _HAS_CUDA
    if _HAS_CUDA is None:
        _HAS_CUDA = torch.cuda.is_available()
    return torch.cuda.current_stream().cuda_stream if _HAS_CUDA else None


def config_struct(cfg: dict) -> Config:
    c = Config()
    for name, _ in Config._fields_:
        if name == "fc_in_features":
            setattr(c, name, int(cfg.get(name, cfg["n_target_layers"] * cfg["target_hidden"])))
        elif name == "rms_eps":
            c.rms_eps = float(cfg[name])
        elif name == "rope_attn_factor":
            c.rope_attn_factor = float(cfg.get(name, 0.0))
        else:
            setattr(c, name, int(cfg.get(name, 0)))
    return c


def yarn_inv_freq(theta: float, head_dim: int, factor: float, beta_fast: float,
                  beta_slow: float, original_max_pos: int):
    """The library's YaRN table (dflash_yarn_inv_freq): (f32 CPU tensor
    [head_dim/2], attention factor for the config's rope_attn_factor)."""
    out = (C.c_float * (head_dim // 2))()
    att = C.c_float()
    _check(lib().dflash_yarn_inv_freq(float(theta), int(head_dim), float(factor),
                                      float(beta_fast), float(beta_slow), int(original_max_pos),
                                      out, C.byref(att)))
    return torch.tensor(list(out), dtype=torch.float32), att.value


def weights_to_device(w: dict, device="cuda") -> dict:
    """Copies the CPU weight dict (synthetic.make_weights) to the device."""
    out = {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: v.to(device) for k, v in lay.items()} for lay in w["layers"]]
    return out


class State:
    def __init__(self, head: "DraftHead", ptr: int):
        self.head, self.ptr = head, ptr


class DraftHead:
    """One draft head (dflash_create). weights=None builds a bookkeeping-only
    head for host tests."""

    def __init__(self, cfg: dict, weights: dict | None):
        L = lib()
        self.cfg = dict(cfg)
        self._cfg_struct = config_struct(cfg)
        self.gamma, self.vocab = int(cfg["gamma"]), int(cfg["vocab"])
        self.bookkeeping_only = weights is None
        wp = None
        if weights is not None:
            keep = []
            lay_ptrs = []
            for lay in weights["layers"]:
                for k in LAYER_KEYS:
                    lay_ptrs.append(lay[k].data_ptr())
            self._layer_arr = (C.c_void_p * len(lay_ptrs))(*lay_ptrs)
            ws = Weights()
            for name in ("embed", "lm_head", "fc", "hidden_norm", "norm", "inv_freq"):
                setattr(ws, name, weights[name].data_ptr())
            if "lm_head_fp8" in weights:
                ws.lm_head_fp8 = weights["lm_head_fp8"].data_ptr()
                ws.lm_head_scale = weights["lm_head_scale"].data_ptr()
            if "lm_head_nvfp4" in weights:
                ws.lm_head_nvfp4 = weights["lm_head_nvfp4"].data_ptr()
                ws.lm_head_nvfp4_scale = weights["lm_head_nvfp4_scale"].data_ptr()
                ws.lm_head_nvfp4_global = float(weights["lm_head_nvfp4_global"])
            if "kv_scale" in weights:
                ws.kv_scale = weights["kv_scale"].data_ptr()
            ws.layers = C.cast(self._layer_arr, C.POINTER(C.c_void_p))
            self._weights = weights          # borrowed by the library: keep alive
            wp = C.byref(ws)
        h = C.c_void_p()
        _check(L.dflash_create(C.byref(self._cfg_struct), wp, C.byref(h)))
        self.ptr = h.value
        self._results = (OK, BOOKKEEPING_ONLY)
        self._outs = {}
        self._batch = {}
        # the cached argument/result arrays serve one call at a time
        self._lock = threading.Lock()

    def close(self):
        if self.ptr:
            lib().dflash_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- trait calls ----------------------------------------------------------
    def propose_batch_max(self) -> int:
        return lib().dflash_propose_batch_max(self.ptr)

    def block_gamma(self) -> int:
        return lib().dflash_block_gamma(self.ptr)

    def alloc_state(self, budget_tokens: int | None = None) -> State:
        p = C.c_void_p()
        _check(lib().dflash_alloc_state(self.ptr, (2 ** 63 - 1) if budget_tokens is None
                                        else int(budget_tokens), C.byref(p)))
        return State(self, p.value)

    def free_state(self, st: State) -> None:
        _check(lib().dflash_free_state(self.ptr, st.ptr))
        st.ptr = None

    def prefill(self, st: State, stack) -> int:
        n = 0 if stack is None else int(stack.shape[0])
        return _check(lib().dflash_prefill(self.ptr, st.ptr, _ptr(stack), n, _stream()),
                      self._results)

    def propose(self, st: State, last_token: int, position: int, new_rows, num_drafts: int,
                bitmask=None, want_conf: bool = True):
        """Returns (drafts, n_out, conf). new_rows: device tensor [n_new, S] or
        None; a pinned CPU tensor is copied to the device first."""
        new_rows = self._to_device(new_rows)
        n_new = 0 if new_rows is None else int(new_rows.shape[0])
        with self._lock:
            out = self._outs.get(num_drafts)
            if out is None:   # result buffers, reused by every call of this width
                out = ((C.c_uint32 * num_drafts)(), C.c_int32(), C.c_float())
                out = out + (C.byref(out[1]), C.byref(out[2]))
                self._outs[num_drafts] = out
            drafts, n_out, conf, n_ref, c_ref = out
            _check(lib().dflash_propose(self.ptr, st.ptr, int(last_token), int(position),
                                        _ptr(new_rows), n_new, int(num_drafts), _ptr(bitmask),
                                        drafts, n_ref, c_ref if want_conf else None, _stream()),
                   self._results)
            return list(drafts), n_out.value, (conf.value if want_conf else None)

    def propose_batch(self, states, last_tokens, positions, new_rows, num_drafts: int,
                      bitmask=None, want_conf: bool = True):
        """Returns a list of (drafts, n_out, conf), or None when declined."""
        n = len(states)
        new_rows = [self._to_device(r) for r in new_rows]
        with self._lock:
            bufs = self._batch.get((n, num_drafts))
            if bufs is None:   # argument and result arrays, reused by every call of this shape
                bufs = ((C.c_void_p * n)(), (C.c_uint32 * n)(), (C.c_int64 * n)(),
                        (C.c_void_p * n)(), (C.c_int32 * n)(), (C.c_uint32 * (n * num_drafts))(),
                        (C.c_int32 * n)(), (C.c_float * n)())
                self._batch[(n, num_drafts)] = bufs
            st_arr, tok, pos, rows, nn, drafts, n_out, conf = bufs
            st_arr[:] = [s.ptr for s in states]
            tok[:] = [int(t) for t in last_tokens]
            pos[:] = [int(p) for p in positions]
            rows[:] = [None if r is None else r.data_ptr() for r in new_rows]
            nn[:] = [0 if r is None else int(r.shape[0]) for r in new_rows]
            rc = _check(lib().dflash_propose_batch(self.ptr, n, st_arr, tok, pos, rows, nn,
                                                   int(num_drafts), _ptr(bitmask), drafts, n_out,
                                                   conf if want_conf else None, _stream()),
                        (OK, DECLINED, BOOKKEEPING_ONLY))
            if rc == DECLINED:
                return None
            d = np.frombuffer(drafts, dtype=np.uint32).reshape(n, num_drafts).tolist()
            no = np.frombuffer(n_out, dtype=np.int32).tolist()
            cf = np.frombuffer(conf, dtype=np.float32).tolist() if want_conf else [None] * n
        return [(d[i], no[i], cf[i]) for i in range(n)]

    def after_verify(self, st: State, num_accepted: int) -> None:
        _check(lib().dflash_after_verify(self.ptr, st.ptr, int(num_accepted)))

    def after_verify_batch(self, states, num_accepted) -> None:
        """after_verify for every state of a propose_batch in one call; on an
        error no state changes."""
        n = len(states)
        st_arr = (C.c_void_p * n)(*[s.ptr for s in states])
        ks = (C.c_int32 * n)(*[int(k) for k in num_accepted])
        _check(lib().dflash_after_verify_batch(self.ptr, n, st_arr, ks))

    def catchup_batch(self, states, rows, first_pos, tokens=None) -> int:
        """[P2]/[P3] catchup_batch: append rows[i] (device [m, S] or None)
        to states[i] at RoPE positions first_pos[i].. (the state's append
        point); tokens[i] (the paired token ids) are range-checked. Returns
        the rows appended."""
        n = len(states)
        rows = [self._to_device(r) for r in rows]
        st_arr = (C.c_void_p * n)(*[s.ptr for s in states])
        ptrs = (C.c_void_p * n)(*[None if r is None else r.data_ptr() for r in rows])
        counts = (C.c_int32 * n)(*[0 if r is None else int(r.shape[0]) for r in rows])
        fp = (C.c_int64 * n)(*[int(f) for f in first_pos])
        keep, tok = [], None
        if tokens is not None:
            tok = (C.c_void_p * n)()
            for i, t in enumerate(tokens):
                if t is not None and len(t) != counts[i]:
                    # the library reads n_rows[i] ids from the array
                    raise DFlashError(-1, f"state {i}: {len(t)} tokens for {counts[i]} rows")
                if t is not None:
                    a = (C.c_uint32 * max(len(t), 1))(*[int(v) for v in t])
                    keep.append(a)
                    tok[i] = C.cast(a, C.c_void_p)
        written = C.c_int64()
        _check(lib().dflash_catchup_batch(self.ptr, n, st_arr, tok, ptrs, counts, fp,
                                          C.byref(written), _stream()), self._results)
        return written.value

    # -- drafter-KV carry across turns -----------------------------------------
    def take_drafter_kv(self, st: State):
        """[P3] take_drafter_kv: (blocks, rows, None), or None when the state
        holds nothing to carry; the state then behaves as fresh."""
        cap = self.debug_pool()[1]
        blocks = (C.c_int32 * max(cap, 1))()
        n, rows = C.c_int32(), C.c_int64()
        rc = _check(lib().dflash_take_drafter_kv(self.ptr, st.ptr, blocks, cap, C.byref(n),
                                                 C.byref(rows)), (OK, DECLINED))
        if rc == DECLINED:
            return None
        return list(blocks[:n.value]), rows.value, None

    def install_drafter_kv(self, st: State, blocks, rows: int, last_pair_key=None) -> bool:
        """[P3] install_drafter_kv into a fresh state; raises on a bad bundle
        (the caller then still owns it)."""
        arr = (C.c_int32 * max(len(blocks), 1))(*[int(b) for b in blocks])
        _check(lib().dflash_install_drafter_kv(self.ptr, st.ptr, arr, len(blocks), int(rows)))
        return True

    def free_drafter_kv(self, blocks) -> None:
        """[P3] free_drafter_kv: release a carried bundle no state owns."""
        arr = (C.c_int32 * max(len(blocks), 1))(*[int(b) for b in blocks])
        _check(lib().dflash_free_drafter_kv(self.ptr, arr, len(blocks)))

    # -- inspection -----------------------------------------------------------
    def debug_state(self, st: State):
        ctx = C.c_int64()
        first = C.c_int32()
        n = lib().dflash_debug_state(st.ptr, C.byref(ctx), C.byref(first), None, 0)
        _check(min(n, 0))
        tab = (C.c_int32 * max(n, 1))()
        lib().dflash_debug_state(st.ptr, C.byref(ctx), C.byref(first), tab, n)
        return ctx.value, first.value, list(tab)[:n]

    def debug_pool(self):
        used, total = C.c_int32(), C.c_int32()
        _check(lib().dflash_debug_pool(self.ptr, C.byref(used), C.byref(total)))
        return used.value, total.value

    def gather_kv(self, st: State, layer: int, pos0: int, n: int):
        nkv, d = self.cfg["num_kv_heads"], self.cfg["head_dim"]
        k = torch.empty((n, nkv, d), dtype=torch.float32, device="cuda")
        v = torch.empty_like(k)
        _check(lib().dflash_debug_gather_kv(self.ptr, st.ptr, layer, pos0, n, k.data_ptr(),
                                            v.data_ptr(), _stream()))
        torch.cuda.current_stream().synchronize()
        return k, v

    def set_graphs(self, enable: bool):
        """Replay captured CUDA graphs (default) or launch kernels one by one."""
        _check(lib().dflash_debug_set_graphs(self.ptr, 1 if enable else 0))

    def set_fault(self, wait_ns: int):
        """Test hook: every GEMM of later proposes aborts after waiting wait_ns
        on a barrier nothing arrives on (0 = off)."""
        _check(lib().dflash_debug_set_fault(self.ptr, int(wait_ns)))

    def set_chain(self, enable: bool):
        """Few-row proposes take the chained single launch (True) or the
        kernel-per-step path (False, the default)."""
        _check(lib().dflash_debug_set_chain(self.ptr, 1 if enable else 0))

    def last_path_chained(self) -> bool:
        return lib().dflash_debug_last_path(self.ptr) == 1

    def debug_rows(self, n_rows: int):
        """(ids, p1) of the last propose's draft rows, sequence-major."""
        ids = (C.c_int32 * max(n_rows, 1))()
        p1 = (C.c_float * max(n_rows, 1))()
        _check(lib().dflash_debug_rows(self.ptr, int(n_rows), ids, p1, _stream()))
        return list(ids)[:n_rows], list(p1)[:n_rows]

    def set_taps(self, x_taps=None, z=None, logits=None):
        self._taps = (x_taps, z, logits)
        _check(lib().dflash_debug_set_taps(self.ptr, _ptr(x_taps), _ptr(z), _ptr(logits)))

    def _to_device(self, t):
        if t is None or t.is_cuda or self.bookkeeping_only:
            return t
        return t.to("cuda", non_blocking=t.is_pinned())
