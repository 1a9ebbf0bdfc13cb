"""Device buffers of a CompKV cache, allocated with PyTorch, driven through the C ABI.

PyTorch provides the device memory and the stream; each method checks its
tensors (device, dtype, shape, contiguity) and passes their addresses to the
library.  Nothing here computes any part of the decode step.
"""
from __future__ import annotations

import torch

from . import compkv as C

BLOCK = 16


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class CompKVCache:
    """A CompKV cache of `num_layers` layers x `batch` sequences on one GPU.

    capacity_tokens: an int (every sequence) or a list (ragged), multiples of 16.
    kv_memory: "device" (the K and V rows in GPU memory, the default) or "host"
        (in page-locked host memory, which the GPU reads over its chip-to-chip
        link; the summaries, the scratch and everything else stay in GPU memory).
    """

    def __init__(self, *, num_layers, batch, num_kv_heads, group_size, head_dim, r,
                 budget_tokens, capacity_tokens, device="cuda", variant=0, kv_memory="device"):
        self.device = torch.device(device)
        if self.device.type != "cuda":
            raise RuntimeError("CompKVCache lives in GPU memory; the library has no CPU path")
        if self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        caps = [capacity_tokens] * batch if isinstance(capacity_tokens, int) else list(capacity_tokens)
        self.cfg = C.make_config(num_layers, batch, num_kv_heads, group_size, head_dim, r,
                                 budget_tokens, capacity_tokens=caps, variant=variant)
        self.variant = variant
        self.num_layers, self.batch, self.Hkv, self.G = num_layers, batch, num_kv_heads, group_size
        self.d, self.r, self.K = head_dim, r, budget_tokens // BLOCK
        self.caps = caps
        self.max_cap_blocks = max(caps) // BLOCK
        rows = C.compkv_rows_per_layer(self.cfg)
        if rows <= 0:
            raise C.CompKVError(2, C.compkv_last_error())
        self.rows_per_layer = rows
        total = rows * num_layers
        dev = self.device
        if kv_memory not in ("device", "host"):
            raise ValueError(f"kv_memory must be 'device' or 'host', got {kv_memory!r}")
        self.kv_memory = kv_memory
        if kv_memory == "host":
            self.k = torch.zeros((total, BLOCK, head_dim), dtype=torch.bfloat16, pin_memory=True)
            self.v = torch.zeros((total, BLOCK, head_dim), dtype=torch.bfloat16, pin_memory=True)
        else:
            self.k = torch.zeros((total, BLOCK, head_dim), dtype=torch.bfloat16, device=dev)
            self.v = torch.zeros((total, BLOCK, head_dim), dtype=torch.bfloat16, device=dev)
        self.kbar = torch.zeros((total, head_dim), dtype=torch.float32, device=dev)
        self.vbar = torch.zeros((total, head_dim), dtype=torch.float32, device=dev)
        self.dbar = torch.zeros((total, r), dtype=torch.float32, device=dev)
        self.seq_len = torch.zeros((num_layers, batch), dtype=torch.int32, device=dev)
        nbytes = C.compkv_scratch_bytes(self.cfg)
        self.scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.bufs = C.compkv_buffers(self.k.data_ptr(), self.v.data_ptr(), self.kbar.data_ptr(),
                                     self.vbar.data_ptr(), self.dbar.data_ptr(),
                                     self.seq_len.data_ptr(), self.scratch.data_ptr(), nbytes)
        with torch.cuda.device(dev):
            self.ctx = C.compkv_init(self.cfg, self.bufs)

    # ------------------------------------------------------------------ layout
    def rows(self, layer, seq, head):
        """(first row, capacity in blocks) of a (layer, sequence, head)."""
        return C.compkv_row_offset(self.ctx, layer, seq, head)

    def token_view(self, layer, seq, head):
        """Views [capacity_tokens, d] of the K and V tokens of one (layer, sequence, head)."""
        r0, cap = self.rows(layer, seq, head)
        return (self.k[r0:r0 + cap].view(cap * BLOCK, self.d),
                self.v[r0:r0 + cap].view(cap * BLOCK, self.d))

    def summary_view(self, layer, seq, head):
        r0, cap = self.rows(layer, seq, head)
        return self.kbar[r0:r0 + cap], self.dbar[r0:r0 + cap], self.vbar[r0:r0 + cap]

    # ------------------------------------------------------------------ checks
    def _t(self, t, name, dtype, shape):
        if t.device != self.device or t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dtype} {tuple(shape)} on {self.device}, "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")
        return t.data_ptr()

    def _q(self, q):
        return self._t(q, "q", torch.float32, (self.batch, self.Hkv * self.G, self.d))

    def _kv(self, t, name):
        return self._t(t, name, torch.bfloat16, (self.batch, self.Hkv, self.d))

    def new_sel(self):
        return torch.empty((self.batch, self.Hkv, self.K), dtype=torch.int32, device=self.device)

    def new_out(self):
        return torch.empty((self.batch, self.Hkv * self.G, self.d), dtype=torch.float32, device=self.device)

    # ------------------------------------------------------------------ calls
    def prefill(self, layer, lens):
        C.compkv_prefill(self.ctx, layer, [int(x) for x in lens], _stream(self.device))

    def append(self, layer, k_new, v_new):
        C.compkv_append(self.ctx, layer, self._kv(k_new, "k_new"), self._kv(v_new, "v_new"),
                        _stream(self.device))

    def score_select(self, layer, q, sel=None, scores=None):
        sel = self.new_sel() if sel is None else sel
        sp = 0
        if scores is not None:
            sp = self._t(scores, "scores", torch.float32, (self.batch, self.Hkv, self.max_cap_blocks))
        C.compkv_score_select(self.ctx, layer, self._q(q),
                              self._t(sel, "sel", torch.int32, (self.batch, self.Hkv, self.K)),
                              sp, _stream(self.device))
        return sel

    def attend(self, layer, q, sel, out=None):
        out = self.new_out() if out is None else out
        C.compkv_attend(self.ctx, layer, self._q(q),
                        self._t(sel, "sel", torch.int32, (self.batch, self.Hkv, self.K)),
                        self._t(out, "out", torch.float32, (self.batch, self.Hkv * self.G, self.d)),
                        _stream(self.device))
        return out

    def decode(self, layer, q, k_new, v_new, out=None, sel=None):
        out = self.new_out() if out is None else out
        sp = 0 if sel is None else self._t(sel, "sel", torch.int32, (self.batch, self.Hkv, self.K))
        C.compkv_decode(self.ctx, layer, self._q(q), self._kv(k_new, "k_new"), self._kv(v_new, "v_new"),
                        self._t(out, "out", torch.float32, (self.batch, self.Hkv * self.G, self.d)),
                        sp, _stream(self.device))
        return out

    def prepared_decode(self):
        """A compkv_decode bound to this cache's context and the current stream:
        call it with (layer, q_ptr, k_ptr, v_ptr, out_ptr, sel_ptr) as plain
        device addresses; no per-call tensor checks."""
        return C.PreparedDecode(self.ctx, _stream(self.device))

    def decode_host(self, layer, q, k_new, v_new, out, sel=None):
        """compkv_decode_host on CPU tensors (q fp32 [B][Hq][d], k_new/v_new bf16
        [B][Hkv][d], out fp32 [B][Hq][d], sel int32 [B][Hkv][K] or None); returns
        when out is filled.  Page-locked tensors are read and written by the
        kernels directly; others are copied."""
        for t, name in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (out, "out")):
            if t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU tensor")
        C.compkv_decode_host(self.ctx, layer, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), out.data_ptr(),
                             0 if sel is None else sel.data_ptr(), _stream(self.device))
        return out

    def device_status(self) -> int:
        return C.compkv_device_status(self.ctx, _stream(self.device))

    def selftest_wait_timeout(self):
        C.compkv_selftest_wait_timeout(self.ctx, _stream(self.device))

    def launch_count(self) -> int:
        return C.compkv_launch_count(self.ctx)

    def profile(self, enable):
        C.compkv_profile_enable(self.ctx, enable)

    def profile_read(self, family):
        return C.compkv_profile_read(self.ctx, family)

    def close(self):
        if getattr(self, "ctx", None):
            C.compkv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
