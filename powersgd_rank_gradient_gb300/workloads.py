"""Seeded synthetic workloads: bucket shape lists and gradient generators.

This module holds no PowerSGD arithmetic.  It is shared by the tests (which
feed the same arrays to the CUDA library and to the fp64 oracle) and by the
benchmark.  Gradients are Gaussian stand-ins for real ones; no dataset or
trained weight is involved.

Shape lists (bucket order, one flat bucket per replica):
* ResNet-50: conv1, four bottleneck stages [3, 4, 6, 3] of widths
  [64, 128, 256, 512] (expansion 4, a downsample conv in each stage's first
  block), two 1-D batch-norm tensors after every conv, fc 1000x2048 + bias.
* BERT-large: word embedding 30522x1024, position embedding 512x1024, the
  embedding LayerNorm pair, then 24 layers of Q/K/V/O 1024x1024 (+ bias),
  two LayerNorm vectors, FFN 4096x1024 (+ bias) and 1024x4096 (+ bias), two
  LayerNorm vectors.
* GPT-2-XL: wte 50257x1600, 48 layers of ln_1 pair, QKV 1600x4800 (+ bias),
  proj 1600x1600 (+ bias), ln_2 pair, MLP 1600x6400 (+ bias) and 6400x1600
  (+ bias), final LayerNorm pair.
"""

from __future__ import annotations

import math

import numpy as np


def resnet50_shapes():
    shapes = [(64, 3, 7, 7), (64,), (64,)]
    inp = 64
    for width, blocks in zip([64, 128, 256, 512], [3, 4, 6, 3]):
        for b in range(blocks):
            shapes += [(width, inp, 1, 1), (width,), (width,),
                       (width, width, 3, 3), (width,), (width,),
                       (4 * width, width, 1, 1), (4 * width,), (4 * width,)]
            if b == 0:
                shapes += [(4 * width, inp, 1, 1), (4 * width,), (4 * width,)]
            inp = 4 * width
    shapes += [(1000, 2048), (1000,)]
    return shapes


def bert_large_shapes(layers=24, embeddings=True):
    shapes = [(30522, 1024), (512, 1024), (1024,), (1024,)] if embeddings else []
    for _ in range(layers):
        shapes += [(1024, 1024), (1024,)] * 4
        shapes += [(1024,), (1024,), (4096, 1024), (4096,), (1024, 4096), (1024,),
                   (1024,), (1024,)]
    return shapes


def gpt2_xl_shapes(layers=48, embeddings=True):
    shapes = [(50257, 1600)] if embeddings else []
    for _ in range(layers):
        shapes += [(1600,), (1600,), (1600, 4800), (4800,), (1600, 1600), (1600,),
                   (1600,), (1600,), (1600, 6400), (6400,), (6400, 1600), (1600,)]
    if embeddings:
        shapes += [(1600,), (1600,)]
    return shapes


def numel(shape):
    n = 1
    for d in shape:
        n *= int(d)
    return n


def bucket_numel(shapes):
    return sum(numel(s) for s in shapes)


def replica_seed(replica, step):
    """Per-(replica, step) seed of the gradient stream: 1000*w + step."""
    return 1000 * replica + step


def heavy_rows(shape, fraction, seed):
    """Row indices (of the (shape[0], -1) view) chosen by a seeded permutation:
    ceil(fraction * rows) of them."""
    rows = int(shape[0])
    k = int(math.ceil(fraction * rows))
    rng = np.random.default_rng(seed)
    return np.sort(rng.permutation(rows)[:k])


def gaussian_bucket_np(shapes, std, seed, heavy_fraction=0.0, heavy_scale=100.0,
                       heavy_seed=12345, dtype=np.float32):
    """One replica's flat bucket on the host: N(0, std) entries drawn with
    numpy's PCG64 from ``seed``; optionally a seeded ``heavy_fraction`` of the
    rows of every >=2-D tensor multiplied by ``heavy_scale`` (the same rows for
    every replica and step)."""
    rng = np.random.default_rng(seed)
    flat = (rng.standard_normal(bucket_numel(shapes)) * std).astype(np.float32)
    if heavy_fraction > 0.0:
        off = 0
        for t, s in enumerate(shapes):
            n = numel(s)
            if len(s) >= 2:
                view = flat[off:off + n].reshape(s[0], -1)
                view[heavy_rows(s, heavy_fraction, heavy_seed + t)] *= heavy_scale
            off += n
    return flat.astype(dtype)


def standard_normal_np(shape, seed):
    """float32 N(0,1) sample (numpy PCG64 ``default_rng(seed)``)."""
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def gaussian_bucket_torch(shapes, std, seed, device, heavy_fraction=0.0,
                          heavy_scale=100.0, heavy_seed=12345, out=None):
    """Device-side version of :func:`gaussian_bucket_np` for full-size buckets
    (``torch.Generator`` on the device; not bit-equal to the numpy stream)."""
    import torch

    n = bucket_numel(shapes)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=device)
    out.normal_(mean=0.0, std=float(std), generator=gen)
    if heavy_fraction > 0.0:
        off = 0
        for t, s in enumerate(shapes):
            k = numel(s)
            if len(s) >= 2:
                view = out[off:off + k].view(s[0], -1)
                idx = torch.from_numpy(heavy_rows(s, heavy_fraction, heavy_seed + t)).to(device)
                view[idx] *= heavy_scale
            off += k
    return out


WORKLOADS = {
    # name: (shapes fn, W, r, min_compression_rate, std, heavy_fraction, batch_same_shape, steps)
    "resnet50": dict(shapes=resnet50_shapes, world_size=4, rank=2, mcr=2.0, std=1e-3,
                     heavy=0.0, batch_same_shape=False, steps=5),
    "bert-large": dict(shapes=bert_large_shapes, world_size=8, rank=4, mcr=2.0, std=1e-3,
                       heavy=0.01, batch_same_shape=True, steps=10),
    "gpt2-xl": dict(shapes=gpt2_xl_shapes, world_size=2, rank=8, mcr=2.0, std=1e-3,
                    heavy=0.0, batch_same_shape=False, steps=5),
}
