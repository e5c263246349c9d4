"""Oracle-side model weights built from the seeded raw tensors.

The raw fp32 weights come from ``synth``; this side encodes them with the
oracle's own int4 encoder.  Nothing here touches the CUDA library.
"""

import functools

import numpy as np
import torch

import oracle
import synth


def quant(raw, g):
    return oracle.quantize_w4(raw.detach().cpu().numpy().astype(np.float32), g)


def bf16_bits(t):
    """uint16 bit patterns of a bf16 torch tensor."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_config(cfg, layers=None, max_streams=8, ctx_cap=None):
    return oracle.OracleConfig(
        hidden=cfg["hidden"], q_heads=cfg["q_heads"], kv_heads=cfg["kv_heads"],
        head_dim=cfg["head_dim"], experts=cfg["experts"], top_k=cfg["top_k"],
        ffn=cfg["ffn"], group=cfg["group"], vocab=cfg["vocab"],
        layers=layers if layers is not None else cfg["layers"],
        rope_base=cfg["rope_base"], ctx_cap=ctx_cap or cfg.get("ctx_cap", 4096),
        max_streams=max_streams)


def oracle_weights(cfg_name, cfg, layers, device="cpu"):
    """Weights dict for ``oracle.model_step``; experts are encoded on demand."""
    g = cfg["group"]

    def layer_weights(l):
        @functools.lru_cache(maxsize=None)
        def expert(e):
            return {n: quant(synth.model_tensor(cfg_name, cfg, n, l, e, device), g)
                    for n in ("wg", "wu", "wd")}
        return {
            "wqkv": quant(synth.model_tensor(cfg_name, cfg, "wqkv", l, device=device), g),
            "wo": quant(synth.model_tensor(cfg_name, cfg, "wo", l, device=device), g),
            "wr": synth.model_tensor(cfg_name, cfg, "wr", l, device=device).cpu().numpy(),
            "expert": expert,
        }

    embed = synth.model_tensor(cfg_name, cfg, "embed", device=device).cpu()
    lm = synth.model_tensor(cfg_name, cfg, "lm_head", device=device)
    return {
        "embed_row": lambda t: embed[t].to(torch.float64).numpy(),
        "layers": [layer_weights(l) for l in range(layers)],
        "lm_head_bits": bf16_bits(lm),
    }
