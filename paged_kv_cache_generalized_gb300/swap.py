"""Layer-by-layer swap-in of KV blocks from the CPU tier, overlapped with the attention of the
layers already in place ("Stateful Large Language Model Serving with Pensieve", sections
"GPU-CPU 2層キャッシュ構造" and "パイプライン化されたswap-in": a layer's KV is used only by that
layer's attention, so layer i starts as soon as its own blocks have landed while layer i+1's
transfer runs).

This module is stream and event orchestration only: every byte is moved by the library's
``block_copy`` kernel or by a plain copy-engine transfer of contiguous host memory.  Two
transfer paths:

``staged``  each layer's swapped blocks sit contiguously in the page-locked host pool, so the
            copy engine moves them in one large transfer per layer into a device staging slot
            (no SM is involved, and large transfers are what the host link needs: "KVキャッシュ
            管理の教科書" 第14章), and ``block_copy`` then scatters the staged blocks to their pool
            slots at HBM speed.  Two staging slots alternate between layers.
``gather``  ``block_copy`` reads every block straight from the host pool over the host link, on
            a copy stream, with ``max_ctas`` bounding the SMs it takes from the attention beside it.

Pools are ``[L, P, num_blocks, *block]`` with P planes per layer (K and V); the host pool holds
``Hn`` swapped blocks per layer and plane, host block i going to device block ``dev_blocks[i]``.
"""
from __future__ import annotations

import torch

from . import pagedkv as _pk


class LayerSwapIn:
    """Issues the swap-in of layer l's blocks ahead of layer l's attention.

    Usage (on the caller's current stream, which runs the attention)::

        sw = LayerSwapIn(host_pool, dev_pool, dev_blocks, mode="staged")
        sw.start()
        for l in range(L):
            sw.wait(l)          # layer l's blocks are in place for work issued after this call
            attention(l)
            sw.advance(l)       # lets the transfer of layer l + 2 reuse layer l's staging slot
    """

    def __init__(self, host_pool: torch.Tensor, dev_pool: torch.Tensor, dev_blocks: torch.Tensor,
                 mode: str = "staged", max_ctas: int = 32, copy_stream=None):
        if mode not in ("staged", "gather"):
            raise ValueError("mode must be 'staged' or 'gather'")
        if host_pool.dim() < 4 or dev_pool.dim() != host_pool.dim():
            raise ValueError("pools must be [L, planes, num_blocks, ...]")
        if host_pool.shape[:2] != dev_pool.shape[:2] or host_pool.shape[3:] != dev_pool.shape[3:]:
            raise ValueError("host and device pools disagree on layers, planes or block shape")
        if not host_pool.is_pinned():
            raise ValueError("the host pool must be page-locked")
        if dev_blocks.dtype != torch.int64 or dev_blocks.numel() != host_pool.shape[2]:
            raise ValueError("dev_blocks must be int64 with one entry per host block")
        self.host, self.dev, self.mode, self.max_ctas = host_pool, dev_pool, mode, int(max_ctas)
        self.L = host_pool.shape[0]
        self.compute = torch.cuda.current_stream(dev_pool.device)
        self.copy = copy_stream or torch.cuda.Stream(dev_pool.device, priority=-1)
        hn = host_pool.shape[2]
        idx = torch.arange(hn, dtype=torch.int64, device=dev_pool.device)
        dst = dev_blocks.to(dev_pool.device)
        self.pairs_staged = torch.stack([idx, dst], 1).contiguous()
        self.pairs_gather = self.pairs_staged      # host index -> device block, same table
        if mode == "staged":
            self.staging = torch.empty((2,) + tuple(host_pool.shape[1:]), dtype=dev_pool.dtype,
                                       device=dev_pool.device)
        self.copied = [torch.cuda.Event() for _ in range(self.L)]
        self.freed = [torch.cuda.Event() for _ in range(self.L)]

    def _issue(self, layer: int):
        with torch.cuda.stream(self.copy):
            if self.mode == "staged":
                if layer >= 2:
                    self.copy.wait_event(self.freed[layer - 2])
                self.staging[layer % 2].copy_(self.host[layer], non_blocking=True)
            else:
                _pk.block_copy(self.host[layer], self.dev[layer], self.pairs_gather, stream=self.copy,
                               max_ctas=self.max_ctas)
            self.copied[layer].record(self.copy)

    def start(self):
        """Issues the first transfers (layers 0 and 1), after the work already queued on the
        compute stream (which may still read the blocks and staging slots being refilled)."""
        self.copy.wait_stream(self.compute)
        for layer in range(min(2, self.L)):
            self._issue(layer)

    def wait(self, layer: int):
        """Makes the compute stream wait for layer ``layer``'s blocks (and, on the staged path,
        scatters them from the staging slot into the pool on the compute stream)."""
        self.compute.wait_event(self.copied[layer])
        if self.mode == "staged":
            _pk.block_copy(self.staging[layer % 2], self.dev[layer], self.pairs_staged,
                           stream=self.compute)
            self.freed[layer].record(self.compute)

    def advance(self, layer: int):
        """Issues the transfer two layers ahead (the staging slot of ``layer`` is free once its
        scatter, already on the compute stream, has run)."""
        if layer + 2 < self.L:
            self._issue(layer + 2)

    def run(self, attention=None):
        """The whole schedule: for each layer, wait for its blocks, then ``attention(layer)``."""
        self.start()
        for layer in range(self.L):
            self.wait(layer)
            if attention is not None:
                attention(layer)
            self.advance(layer)


def swap_out_pairs(dev_blocks: torch.Tensor) -> torch.Tensor:
    """The (device block, host block) table of ``swap_out``: device block ``dev_blocks[i]`` goes
    to host block i."""
    idx = torch.arange(dev_blocks.numel(), dtype=torch.int64, device=dev_blocks.device)
    return torch.stack([dev_blocks.to(torch.int64), idx], 1).contiguous()


def swap_out(dev_pool: torch.Tensor, host_pool: torch.Tensor, pairs: torch.Tensor, stream=None,
             max_ctas: int = 0):
    """Evicts blocks to the CPU tier: for every layer and plane, ``block_copy`` gathers the device
    blocks of ``pairs`` (see ``swap_out_pairs``) and writes them over the host link into the
    page-locked host pool."""
    for layer in range(dev_pool.shape[0]):
        _pk.block_copy(dev_pool[layer], host_pool[layer], pairs, stream=stream, max_ctas=max_ctas)
