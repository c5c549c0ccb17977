"""Convenience wrapper around the C ABI for callers that hold KV in torch tensors.

PyTorch provides device memory and streams only; every step runs in libkvc.so.
A Codec owns a plan and a workspace (the "persistent runtime scratch" of "Beyond
Compression Ratio: High-Throughput KV Compression for Disaggregated LLM Serving",
§4.2) and reuses both across requests.
"""
from __future__ import annotations

import torch

from . import kvc


class Codec:
    def __init__(self, profile: kvc.Profile, shape: kvc.Shape, device="cuda"):
        self.device = torch.device(device)
        self.profile, self.shape = profile, shape
        self.plan = kvc.Plan(profile, shape)
        self.workspace = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8, device=self.device)
        self.d_size = torch.zeros(1, dtype=torch.int64, device=self.device)

    def _stream(self) -> int:
        return torch.cuda.current_stream(self.device).cuda_stream

    def new_stream_buffer(self) -> torch.Tensor:
        return torch.empty(self.plan.max_stream_bytes, dtype=torch.uint8, device=self.device)

    def new_payload_buffer(self) -> torch.Tensor:
        return torch.empty(max(self.plan.payload_bytes, 16), dtype=torch.uint8, device=self.device)

    def encode(self, k_layers, v_layers, block_table=None, out: torch.Tensor | None = None):
        """Enqueue an encode; returns the stream buffer (size via `query()`)."""
        out = self.new_stream_buffer() if out is None else out
        kv = kvc.KVRef.from_tensors(k_layers, v_layers, block_table)
        kvc.kvc_encode(self.plan, kv, out.data_ptr(), out.numel(), self.workspace.data_ptr(),
                       self.workspace.numel(), self.d_size.data_ptr(), self._stream())
        return out

    def decode(self, stream: torch.Tensor, stream_bytes: int, k_layers, v_layers, block_table=None):
        kv = kvc.KVRef.from_tensors(k_layers, v_layers, block_table)
        kvc.kvc_decode(self.plan, stream.data_ptr(), stream_bytes, kv, self.workspace.data_ptr(),
                       self.workspace.numel(), self._stream())

    def quantize(self, k_layers, v_layers, block_table=None, out: torch.Tensor | None = None):
        out = self.new_payload_buffer() if out is None else out
        kv = kvc.KVRef.from_tensors(k_layers, v_layers, block_table)
        kvc.kvc_quantize(self.plan, kv, out.data_ptr(), self.workspace.data_ptr(), self.workspace.numel(),
                         self._stream())
        return out

    def lossless_encode(self, payload: torch.Tensor, out: torch.Tensor | None = None):
        out = self.new_stream_buffer() if out is None else out
        kvc.kvc_lossless_encode(self.plan, payload.data_ptr(), out.data_ptr(), out.numel(),
                                self.workspace.data_ptr(), self.workspace.numel(), self.d_size.data_ptr(),
                                self._stream())
        return out

    def lossless_decode(self, stream: torch.Tensor, stream_bytes: int, out: torch.Tensor | None = None):
        out = self.new_payload_buffer() if out is None else out
        kvc.kvc_lossless_decode(self.plan, stream.data_ptr(), stream_bytes, out.data_ptr(),
                                self.workspace.data_ptr(), self.workspace.numel(), self._stream())
        return out

    def dequantize(self, payload: torch.Tensor, k_layers, v_layers, block_table=None):
        kv = kvc.KVRef.from_tensors(k_layers, v_layers, block_table)
        kvc.kvc_dequantize(self.plan, payload.data_ptr(), kv, self.workspace.data_ptr(), self.workspace.numel(),
                           self._stream())

    def query(self):
        """(status, stream_bytes, flags); synchronizes the current stream."""
        return kvc.kvc_query(self.workspace.data_ptr(), self._stream())
