"""Thin Python binding of the C ABI (``include/spec_verify.h``).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their device pointers and the current CUDA stream are handed to
the library, and every step of the verification pass runs in the library's
CUDA kernels. PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _native

F32, BF16 = 0, 1
STOCHASTIC, GREEDY, FLY = 0, 1, 2
MODES = {"stochastic": STOCHASTIC, "greedy": GREEDY, "fly": FLY}

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_CUDA = 3
SPEC_ERR_TIMEOUT = 4
SPEC_ERR_BAD_ROW = 5
SPEC_ERR_BAD_TOKEN = 6
SPEC_ERR_BAD_TEMPERATURE = 7
SPEC_ERR_INDEX = 8
MAX_K = 31
MAX_V = 1 << 20


class SpecError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"spec_verify error {code}: {msg}")
        self.code = code


def _check(rc: int):
    if rc != SPEC_OK:
        raise SpecError(rc, _native.last_error())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream: Optional[torch.cuda.Stream], device: torch.device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _row_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() != 3:
        raise ValueError(f"{name} must be 3-D [B, rows, V]")
    if t.stride(2) != 1:
        raise ValueError(f"{name}: the vocabulary axis must be contiguous")
    # rows of one sequence and successive sequences must be evenly spaced
    if t.stride(0) != t.stride(1) * t.shape[1] and t.shape[0] > 1:
        raise ValueError(f"{name}: rows must be evenly spaced (stride[0] == stride[1] * shape[1])")
    return int(t.stride(1))


def make_params(B, K, V, dtype, mode="stochastic", fly_theta=0.3, fly_window=6,
                t_row_stride=0, d_row_stride=0) -> _native.VerifyParams:
    p = _native.VerifyParams()
    p.B, p.K, p.V = int(B), int(K), int(V)
    p.dtype = int(dtype)
    p.mode = MODES[mode] if isinstance(mode, str) else int(mode)
    p.fly_window = int(fly_window)
    p.fly_theta = float(fly_theta)
    p.reserved = 0
    p.t_row_stride = int(t_row_stride)
    p.d_row_stride = int(d_row_stride)
    return p


def workspace_size(params: _native.VerifyParams) -> int:
    return int(_native.lib().spec_workspace_size(ctypes.byref(params)))


class Workspace:
    """Device scratch for spec_verify / spec_confidence, grown on demand."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else None
        self.buf = None

    def get(self, nbytes: int, device: torch.device) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            # 16-byte alignment: torch allocations are 256-byte aligned
            self.buf = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        return self.buf


_default_ws = {}


def _ws_for(ws: Optional[Workspace], nbytes: int, device: torch.device) -> torch.Tensor:
    if ws is None:
        ws = _default_ws.setdefault(device, Workspace(device))
    return ws.get(nbytes, device)


def verify(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor],
           draft_tokens: torch.Tensor, uniforms: Optional[torch.Tensor], mode: str = "stochastic",
           fly_theta: float = 0.3, fly_window: int = 6, est_params: Optional[torch.Tensor] = None,
           want_pos_stats: bool = False, want_feature: bool = False, want_conf: bool = False,
           out: Optional[dict] = None, workspace: Optional[Workspace] = None,
           stream: Optional[torch.cuda.Stream] = None, draft_len: Optional[torch.Tensor] = None,
           inv_temperature: Optional[torch.Tensor] = None, top_p: Optional[float] = None) -> dict:
    """Run spec_verify (spec_verify_ragged when ``draft_len`` [B] int32 gives
    the drafts verified per sequence of a pruned batch; spec_verify_temperature
    when ``inv_temperature`` [B] float32 gives 1/T per sequence;
    spec_verify_top_p when ``top_p`` in (0, 1] is given). Returns a dict with
    ``out_tokens`` [B,K+1] int32 and ``accepted_len`` [B] int32, plus
    ``pos_stats`` [B,K+1,4], ``feature`` [B,K] and ``conf`` [B,K] (float32)
    when requested. ``out`` may supply preallocated output tensors under the
    same keys."""
    zt = target_logits
    if not zt.is_cuda:
        raise ValueError("target_logits must be a CUDA tensor")
    dev = zt.device
    B, K1, V = zt.shape
    K = K1 - 1
    dt = _dtype_code(zt)
    ts = _row_stride(zt, "target_logits")
    ds = 0
    if draft_logits is not None:
        if draft_logits.dtype != zt.dtype or tuple(draft_logits.shape) != (B, K, V):
            raise ValueError("draft_logits must match target_logits' dtype and be [B, K, V]")
        if draft_logits.device != dev:
            raise ValueError("draft_logits must be on the target's device")
        ds = _row_stride(draft_logits, "draft_logits")
    x = draft_tokens
    if x.dtype != torch.int32 or tuple(x.shape) != (B, K) or not x.is_contiguous() or x.device != dev:
        raise ValueError("draft_tokens must be a contiguous int32 [B, K] tensor on the logits' device")
    if uniforms is not None:
        if (uniforms.dtype != torch.float32 or tuple(uniforms.shape) != (B, K + 1)
                or not uniforms.is_contiguous() or uniforms.device != dev):
            raise ValueError("uniforms must be a contiguous float32 [B, K+1] tensor on the logits' device")
    if est_params is not None:
        if est_params.dtype != torch.float32 or est_params.numel() != K + 1 or est_params.device != dev:
            raise ValueError("est_params must be a float32 [K+1] tensor on the logits' device")
    if draft_len is not None:
        if (draft_len.dtype != torch.int32 or tuple(draft_len.shape) != (B,) or not draft_len.is_contiguous()
                or draft_len.device != dev):
            raise ValueError("draft_len must be a contiguous int32 [B] tensor on the logits' device")
    if inv_temperature is not None:
        if (inv_temperature.dtype != torch.float32 or tuple(inv_temperature.shape) != (B,)
                or not inv_temperature.is_contiguous() or inv_temperature.device != dev):
            raise ValueError("inv_temperature must be a contiguous float32 [B] tensor on the logits' device")
    o = dict(out or {})
    if "out_tokens" not in o:
        o["out_tokens"] = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if "accepted_len" not in o:
        o["accepted_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
    if want_pos_stats and "pos_stats" not in o:
        o["pos_stats"] = torch.empty((B, K + 1, 4), dtype=torch.float32, device=dev)
    if want_feature and "feature" not in o:
        o["feature"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    if want_conf and "conf" not in o:
        o["conf"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    p = make_params(B, K, V, dt, mode, fly_theta, fly_window, ts, ds)
    L = _native.lib()
    nbytes = int(L.spec_workspace_size(ctypes.byref(p)))
    if nbytes == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, _native.last_error())
    ws = _ws_for(workspace, nbytes, dev)
    if top_p is not None:
        rc = L.spec_verify_top_p(ctypes.byref(p), _ptr(zt), _ptr(draft_logits), _ptr(x), _ptr(draft_len),
                                 _ptr(inv_temperature), ctypes.c_float(top_p), _ptr(uniforms),
                                 _ptr(o["out_tokens"]), _ptr(o["accepted_len"]), _ptr(o.get("pos_stats")),
                                 _ptr(est_params), _ptr(o.get("feature")), _ptr(o.get("conf")), _ptr(ws),
                                 ctypes.c_size_t(ws.numel()), _stream_ptr(stream, dev))
    elif inv_temperature is not None:
        rc = L.spec_verify_temperature(ctypes.byref(p), _ptr(zt), _ptr(draft_logits), _ptr(x), _ptr(draft_len),
                                       _ptr(inv_temperature), _ptr(uniforms), _ptr(o["out_tokens"]),
                                       _ptr(o["accepted_len"]), _ptr(o.get("pos_stats")), _ptr(est_params),
                                       _ptr(o.get("feature")), _ptr(o.get("conf")), _ptr(ws),
                                       ctypes.c_size_t(ws.numel()), _stream_ptr(stream, dev))
    elif draft_len is None:
        rc = L.spec_verify(ctypes.byref(p), _ptr(zt), _ptr(draft_logits), _ptr(x), _ptr(uniforms),
                           _ptr(o["out_tokens"]), _ptr(o["accepted_len"]), _ptr(o.get("pos_stats")),
                           _ptr(est_params), _ptr(o.get("feature")), _ptr(o.get("conf")),
                           _ptr(ws), ctypes.c_size_t(ws.numel()), _stream_ptr(stream, dev))
    else:
        rc = L.spec_verify_ragged(ctypes.byref(p), _ptr(zt), _ptr(draft_logits), _ptr(x), _ptr(draft_len),
                                  _ptr(uniforms), _ptr(o["out_tokens"]), _ptr(o["accepted_len"]),
                                  _ptr(o.get("pos_stats")), _ptr(est_params), _ptr(o.get("feature")),
                                  _ptr(o.get("conf")), _ptr(ws), ctypes.c_size_t(ws.numel()),
                                  _stream_ptr(stream, dev))
    _check(rc)
    o["_workspace"] = ws
    return o


def confidence(draft_logits: torch.Tensor, est_params: Optional[torch.Tensor] = None,
               workspace: Optional[Workspace] = None, stream: Optional[torch.cuda.Stream] = None,
               out: Optional[dict] = None):
    """Run spec_confidence: returns (feature [B,K], conf [B,K] or None).
    ``out`` may supply preallocated ``feature`` / ``conf`` tensors."""
    zd = draft_logits
    if not zd.is_cuda:
        raise ValueError("draft_logits must be a CUDA tensor")
    dev = zd.device
    B, K, V = zd.shape
    dt = _dtype_code(zd)
    ds = _row_stride(zd, "draft_logits")
    o = dict(out or {})
    feat = o.get("feature")
    if feat is None:
        feat = torch.empty((B, K), dtype=torch.float32, device=dev)
    conf = None
    if est_params is not None:
        conf = o.get("conf")
        if conf is None:
            conf = torch.empty((B, K), dtype=torch.float32, device=dev)
    for t in (feat, conf):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (B, K) or not t.is_contiguous()
                              or t.device != dev):
            raise ValueError("confidence: out tensors must be contiguous float32 [B, K] on the logits' device")
    L = _native.lib()
    nbytes = int(L.spec_confidence_workspace_size(B, K, V, dt))
    if nbytes == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, _native.last_error())
    ws = _ws_for(workspace, nbytes, dev)
    rc = L.spec_confidence(B, K, V, dt, _ptr(zd), ds, _ptr(est_params), _ptr(feat), _ptr(conf),
                           _ptr(ws), ctypes.c_size_t(ws.numel()), _stream_ptr(stream, dev))
    _check(rc)
    return feat, conf


def estimator_update(feature: torch.Tensor, accepted_len: torch.Tensor, est_params: torch.Tensor,
                     lr: float, want_grad: bool = False, stream: Optional[torch.cuda.Stream] = None,
                     draft_len: Optional[torch.Tensor] = None):
    """Run spec_estimator_update (spec_estimator_update_ragged with
    ``draft_len``) in place on ``est_params``. Returns (grad [K+1], counts
    [K+1]) when ``want_grad``, else None."""
    B, K = feature.shape
    dev = feature.device
    for t, dt_, shp in ((feature, torch.float32, (B, K)), (accepted_len, torch.int32, (B,)),
                        (est_params, torch.float32, (K + 1,))):
        if t.dtype != dt_ or tuple(t.shape) != shp or not t.is_contiguous() or t.device != dev:
            raise ValueError("estimator_update: bad tensor (dtype/shape/device/contiguity)")
    grad = cnt = None
    if want_grad:
        grad = torch.empty(K + 1, dtype=torch.float32, device=dev)
        cnt = torch.empty(K + 1, dtype=torch.int32, device=dev)
    if draft_len is None:
        rc = _native.lib().spec_estimator_update(B, K, _ptr(feature), _ptr(accepted_len), _ptr(est_params),
                                                 float(lr), _ptr(grad), _ptr(cnt), _stream_ptr(stream, dev))
    else:
        _check_draft_len(draft_len, B, dev)
        rc = _native.lib().spec_estimator_update_ragged(B, K, _ptr(feature), _ptr(accepted_len), _ptr(draft_len),
                                                        _ptr(est_params), float(lr), _ptr(grad), _ptr(cnt),
                                                        _stream_ptr(stream, dev))
    _check(rc)
    return (grad, cnt) if want_grad else None


class IrlsState:
    """Device-resident state of one IRLS round (spec_irls_*): 4K+3 doubles,
    zeroed on creation and after every refit."""

    def __init__(self, K: int, device, stream: Optional[torch.cuda.Stream] = None):
        n = _native.lib().spec_irls_state_size(int(K))
        if n == 0:
            raise SpecError(SPEC_ERR_UNSUPPORTED, "IRLS: K must be in [1, 1024]")
        self.K = int(K)
        self.device = torch.device(device)
        self.tensor = torch.empty(n // 8, dtype=torch.float64, device=self.device)
        self.reset(stream)

    def reset(self, stream: Optional[torch.cuda.Stream] = None):
        _check(_native.lib().spec_irls_reset(self.K, _ptr(self.tensor), _stream_ptr(stream, self.device)))

    def parts(self):
        """Views (g [K+1], H_ww [1], H_wb [K], H_bb [K], n [K+1]) of the state."""
        K, t = self.K, self.tensor
        return t[:K + 1], t[K + 1:K + 2], t[K + 2:2 * K + 2], t[2 * K + 2:3 * K + 2], t[3 * K + 2:]


def _check_draft_len(draft_len, B, dev):
    if (draft_len.dtype != torch.int32 or tuple(draft_len.shape) != (B,) or not draft_len.is_contiguous()
            or draft_len.device != dev):
        raise ValueError("draft_len must be a contiguous int32 [B] tensor on the same device")


def irls_accumulate(feature: torch.Tensor, accepted_len: torch.Tensor, est_params: torch.Tensor,
                    state: IrlsState, stream: Optional[torch.cuda.Stream] = None,
                    draft_len: Optional[torch.Tensor] = None):
    """Add one decoding step's labels to an IRLS round (spec_irls_accumulate;
    spec_irls_accumulate_ragged with ``draft_len``)."""
    B, K = feature.shape
    dev = feature.device
    if K != state.K or state.device != dev:
        raise ValueError("irls_accumulate: state does not match K / device")
    for t, dt_, shp in ((feature, torch.float32, (B, K)), (accepted_len, torch.int32, (B,)),
                        (est_params, torch.float32, (K + 1,))):
        if t.dtype != dt_ or tuple(t.shape) != shp or not t.is_contiguous() or t.device != dev:
            raise ValueError("irls_accumulate: bad tensor (dtype/shape/device/contiguity)")
    if draft_len is None:
        rc = _native.lib().spec_irls_accumulate(B, K, _ptr(feature), _ptr(accepted_len), _ptr(est_params),
                                                _ptr(state.tensor), _stream_ptr(stream, dev))
    else:
        _check_draft_len(draft_len, B, dev)
        rc = _native.lib().spec_irls_accumulate_ragged(B, K, _ptr(feature), _ptr(accepted_len), _ptr(draft_len),
                                                       _ptr(est_params), _ptr(state.tensor),
                                                       _stream_ptr(stream, dev))
    _check(rc)


def irls_refit(state: IrlsState, est_params: torch.Tensor, damping: float, want_step: bool = False,
               stream: Optional[torch.cuda.Stream] = None):
    """End an IRLS round: update ``est_params`` in place (spec_irls_refit) and
    zero the state. Returns the applied step [K+1] (fp64) when ``want_step``."""
    K, dev = state.K, state.device
    if est_params.dtype != torch.float32 or tuple(est_params.shape) != (K + 1,) \
            or not est_params.is_contiguous() or est_params.device != dev:
        raise ValueError("irls_refit: bad est_params (dtype/shape/device/contiguity)")
    step = torch.empty(K + 1, dtype=torch.float64, device=dev) if want_step else None
    rc = _native.lib().spec_irls_refit(K, _ptr(state.tensor), _ptr(est_params), float(damping), _ptr(step),
                                       _stream_ptr(stream, dev))
    _check(rc)
    return step


def ngram_draft(ctx: torch.Tensor, lengths: torch.Tensor, n_min: int, n_max: int, K: int,
                stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Prompt-lookup drafts (spec_ngram_draft): returns a dict with
    ``draft_tokens`` [B,K] int32 (-1 padded) and ``draft_len`` [B] int32."""
    B, ld = ctx.shape
    dev = ctx.device
    if ctx.dtype != torch.int32 or not ctx.is_contiguous() or not ctx.is_cuda:
        raise ValueError("ngram_draft: ctx must be a contiguous int32 CUDA tensor [B, ld]")
    if lengths.dtype != torch.int32 or tuple(lengths.shape) != (B,) or lengths.device != dev:
        raise ValueError("ngram_draft: lengths must be an int32 [B] tensor on ctx's device")
    o = {"draft_tokens": torch.empty((B, K), dtype=torch.int32, device=dev),
         "draft_len": torch.empty(B, dtype=torch.int32, device=dev)}
    rc = _native.lib().spec_ngram_draft(B, ld, _ptr(ctx), _ptr(lengths.contiguous()), int(n_min), int(n_max), int(K),
                                        _ptr(o["draft_tokens"]), _ptr(o["draft_len"]), _stream_ptr(stream, dev))
    _check(rc)
    return o


def av_budget(conf: torch.Tensor, draft_cost: torch.Tensor, verify_cost: torch.Tensor,
              want_survival: bool = False, want_objective: bool = False,
              stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Adaptive-verification pruning (spec_av_budget). Returns a dict with
    ``draft_len`` [B] int32 and ``budget`` [1] int32 (device tensors), plus
    ``survival`` [B,K] float32 and ``objective`` [B*K+1] float32 when asked."""
    B, K = conf.shape
    dev = conf.device
    if conf.dtype != torch.float32 or not conf.is_contiguous() or not conf.is_cuda:
        raise ValueError("av_budget: conf must be a contiguous float32 CUDA tensor [B, K]")
    for t in (draft_cost, verify_cost):
        if (t.dtype != torch.float32 or tuple(t.shape) != (B * K + 1,) or not t.is_contiguous()
                or t.device != dev):
            raise ValueError("av_budget: cost tables must be contiguous float32 [B*K+1] on conf's device")
    o = {"draft_len": torch.empty(B, dtype=torch.int32, device=dev),
         "budget": torch.empty(1, dtype=torch.int32, device=dev)}
    if want_survival:
        o["survival"] = torch.empty((B, K), dtype=torch.float32, device=dev)
    if want_objective:
        o["objective"] = torch.empty(B * K + 1, dtype=torch.float32, device=dev)
    rc = _native.lib().spec_av_budget(B, K, _ptr(conf), _ptr(draft_cost), _ptr(verify_cost), _ptr(o["draft_len"]),
                                      _ptr(o["budget"]), _ptr(o.get("survival")), _ptr(o.get("objective")),
                                      _stream_ptr(stream, dev))
    _check(rc)
    return o


def device_status(workspace_tensor: torch.Tensor) -> int:
    """Synchronously read the status word of a workspace (tests, debugging)."""
    v = ctypes.c_int32(-1)
    _check(_native.lib().spec_get_device_status(_ptr(workspace_tensor), ctypes.byref(v)))
    return int(v.value)
