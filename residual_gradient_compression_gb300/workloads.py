"""Seeded synthetic gradient workloads (inputs only: none of the method's arithmetic).

These stand in for the training runs that the AdaComp pages report on (MNIST,
CIFAR10, ImageNet, BN50, Shakespeare; "AdaComp (Adaptive Residual Gradient
Compression)", Claims > Application), which need datasets and trained weights that
are not available. Each workload has the layer shapes, bin lengths and gradient
distributions of one configuration:

* ``fc400k``    one 500x800 FC layer, L_T = 500, dW ~ N(0, 1e-3) fresh each step;
* ``resnet50``  the 53 conv weights of ResNet-50 (L_T = 50, 8-bit codes) and its
  2048x1000 FC (L_T = 500), dW_l ~ N(0, sigma_l), sigma_l = 10^U(-4,-2) per layer;
* ``lstm_fc``   4 LSTM weights 4*1024 x (1024+1024) and six 4096x4096 FC layers,
  L_T = 500, dW = 1e-3 * Student-t(3); 90% of each FC layer's 4096 input rows are
  zero, re-drawn every step;
* ``gpt1p3b``   a 1.3B decoder's tensors (24 layers, d = 2048, FFN 8192, vocab
  50,304), bf16 dW ~ N(0, 1e-3) * 10^U(-1,1) per tensor, L_T chosen by the caller;
* ``flat100m``  one flat 100M-element layer at L_T = 500 for K = 16 learners.

Seeds: 1000*config + 100*step + layer, plus 10^6*learner.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

CONFIG_IDS = {"fc400k": 1, "resnet50": 2, "lstm_fc": 3, "gpt1p3b": 4, "flat100m": 5}


@dataclass(frozen=True)
class Layer:
    name: str
    numel: int
    bin_len: int
    dw_dtype: str  # "f32" or "bf16"
    rows: int = 0  # >0: the layer is viewed as [rows, numel // rows] for row sparsity


def _resnet50_conv_shapes():
    shapes = [("conv1", 64 * 3 * 7 * 7)]
    inp = 64
    for stage, (width, blocks) in enumerate(zip((64, 128, 256, 512), (3, 4, 6, 3))):
        for blk in range(blocks):
            pre = f"layer{stage + 1}.{blk}"
            shapes.append((pre + ".conv1", width * inp))
            shapes.append((pre + ".conv2", width * width * 9))
            shapes.append((pre + ".conv3", 4 * width * width))
            if blk == 0:
                shapes.append((pre + ".downsample", 4 * width * inp))
            inp = 4 * width
    return shapes


def _gpt_shapes():
    d, ffn, vocab, ctx = 2048, 8192, 50304, 2048
    shapes = [("wte", vocab * d), ("wpe", ctx * d)]
    for i in range(24):
        p = f"h{i}."
        shapes += [(p + "ln1.w", d), (p + "ln1.b", d), (p + "qkv.w", 3 * d * d),
                   (p + "qkv.b", 3 * d), (p + "proj.w", d * d), (p + "proj.b", d),
                   (p + "ln2.w", d), (p + "ln2.b", d), (p + "fc1.w", ffn * d),
                   (p + "fc1.b", ffn), (p + "fc2.w", d * ffn), (p + "fc2.b", d)]
    shapes += [("lnf.w", d), ("lnf.b", d)]
    return shapes


def layers(config: str, bin_len: int | None = None) -> list[Layer]:
    if config == "fc400k":
        return [Layer("fc", 500 * 800, 500, "f32")]
    if config == "resnet50":
        out = [Layer(n, k, 50, "f32") for n, k in _resnet50_conv_shapes()]
        return out + [Layer("fc", 1000 * 2048, 500, "f32")]
    if config == "lstm_fc":
        out = [Layer(f"lstm{i}", 4 * 1024 * 2048, 500, "f32") for i in range(4)]
        return out + [Layer(f"fc{i}", 4096 * 4096, 500, "f32", rows=4096) for i in range(6)]
    if config == "gpt1p3b":
        return [Layer(n, k, bin_len or 500, "bf16") for n, k in _gpt_shapes()]
    if config == "flat100m":
        return [Layer("flat", 100_000_000, 500, "f32")]
    raise KeyError(config)


def seed(config: str, step: int, layer: int, learner: int = 0) -> int:
    return 1000 * CONFIG_IDS[config] + 100 * step + layer + 1_000_000 * learner


def _gen(device, s):
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def layer_sigma(config: str, layer: int) -> float:
    """Per-layer scale drawn once per layer (not per step)."""
    g = _gen("cpu", 7_000_000 + 1000 * CONFIG_IDS[config] + layer)
    u = torch.rand(1, generator=g, dtype=torch.float64).item()
    if config == "resnet50":
        return 10.0 ** (-4 + 2 * u)   # log-uniform in [1e-4, 1e-2]
    if config == "gpt1p3b":
        return 1e-3 * 10.0 ** (-1 + 2 * u)  # 1e-3 times log-uniform in [0.1, 10]
    return 1e-3


def gen_dw(config: str, layer_index: int, layer: Layer, step: int, learner: int = 0,
           device="cuda") -> torch.Tensor:
    """dW for one layer and step: fp32, or bf16 rounded to nearest from fp32 draws."""
    g = _gen(device, seed(config, step, layer_index, learner))
    n = layer.numel
    if config == "lstm_fc":
        z = torch.randn(4, n, generator=g, device=device, dtype=torch.float32)
        dw = 1e-3 * z[0] / torch.sqrt((z[1] * z[1] + z[2] * z[2] + z[3] * z[3]) / 3.0)
        if layer.rows:
            keep = torch.rand(layer.rows, generator=g, device=device) < 0.1
            dw = (dw.view(layer.rows, -1) * keep[:, None].to(dw.dtype)).reshape(-1)
    else:
        dw = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        dw.mul_(layer_sigma(config, layer_index))
    if layer.dw_dtype == "bf16":
        return dw.to(torch.bfloat16)
    return dw.contiguous()
