"""CUDA-side model set-up for the tests and the bench.

Raw fp32 weights come from ``synth``, drawn on ``gen_device`` (the oracle
side of a test draws them on the same device so both sides see the same
values); this side encodes them with the library's own int4 encoder
(``bm_w4_quantize``) and loads them into an engine.  Nothing here imports
the oracle.
"""

import torch

import bit_moe_decode_w4a16_gb300 as bm
import synth


def quantize_dev(raw, g, stream=None):
    """Encode an fp32 [N][K] tensor on the GPU; returns (packed uint8, scales fp16)."""
    raw = raw.to("cuda").contiguous().float()
    N, K = raw.shape
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((N, K // g), dtype=torch.float16, device="cuda")
    bm.bm_w4_quantize(raw, N, K, g, packed, scales, stream)
    return packed, scales


def expert_bank(cfg_name, cfg, layer, name, gen_device="cuda"):
    """Packed [E][rows][K/2] and scales [E][rows][K/g] of one expert matrix kind."""
    E, g = cfg["experts"], cfg["group"]
    first = synth.model_tensor(cfg_name, cfg, name, layer, 0, gen_device)
    rows, K = first.shape
    packed = torch.empty((E, rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((E, rows, K // g), dtype=torch.float16, device="cuda")
    for e in range(E):
        raw = first if e == 0 else synth.model_tensor(cfg_name, cfg, name, layer, e, gen_device)
        bm.bm_w4_quantize(raw.to("cuda").contiguous(), rows, K, g, packed[e], scales[e])
    return packed, scales


def layer_weights(cfg_name, cfg, layer, gen_device="cuda"):
    g = cfg["group"]
    wqkv = quantize_dev(synth.model_tensor(cfg_name, cfg, "wqkv", layer, device=gen_device), g)
    wo = quantize_dev(synth.model_tensor(cfg_name, cfg, "wo", layer, device=gen_device), g)
    wr = synth.model_tensor(cfg_name, cfg, "wr", layer, device=gen_device).to("cuda").contiguous()
    wg = expert_bank(cfg_name, cfg, layer, "wg", gen_device)
    wu = expert_bank(cfg_name, cfg, layer, "wu", gen_device)
    wd = expert_bank(cfg_name, cfg, layer, "wd", gen_device)
    return {"wqkv": wqkv[0], "wqkv_s": wqkv[1], "wo": wo[0], "wo_s": wo[1], "wr": wr,
            "wg": wg[0], "wg_s": wg[1], "wu": wu[0], "wu_s": wu[1], "wd": wd[0], "wd_s": wd[1],
            "attn_norm": None, "ffn_norm": None}


def engine_config(cfg, layers, max_streams, ctx_cap, policy=bm.POLICY_AUTO, use_graph=1, prefill_tc=0,
                  persistent_step=0):
    return {"hidden": cfg["hidden"], "q_heads": cfg["q_heads"], "kv_heads": cfg["kv_heads"],
            "head_dim": cfg["head_dim"], "experts": cfg["experts"], "top_k": cfg["top_k"], "ffn": cfg["ffn"],
            "group": cfg["group"], "vocab": cfg["vocab"], "layers": layers, "rope_base": cfg["rope_base"],
            "rms_eps": 1e-6, "max_streams": max_streams, "ctx_cap": ctx_cap, "renorm_topk": 1,
            "kernel_policy": policy, "use_graph": use_graph, "prefill_tc": prefill_tc,
            "persistent_step": persistent_step}


def build_engine(cfg_name, cfg, layers, max_streams, ctx_cap, policy=bm.POLICY_AUTO, use_graph=1,
                 gen_device="cuda", prefill_tc=0, persistent_step=0):
    """An engine with every layer's weights and the embeddings loaded."""
    e = bm.bm_engine_create(engine_config(cfg, layers, max_streams, ctx_cap, policy, use_graph, prefill_tc,
                                          persistent_step))
    for l in range(layers):
        w = layer_weights(cfg_name, cfg, l, gen_device)
        bm.bm_engine_set_layer(e, l, w)
        torch.cuda.synchronize()
        del w
    embed = synth.model_tensor(cfg_name, cfg, "embed", device=gen_device).to("cuda").contiguous()
    lm = synth.model_tensor(cfg_name, cfg, "lm_head", device=gen_device).to("cuda").contiguous()
    bm.bm_engine_set_embeddings(e, embed, lm, None)
    torch.cuda.synchronize()
    return e


def seed_stream(e, cfg_name, cfg, stream, length, layers, gen_device="cuda"):
    """Seed one slot with the stream's synthetic K/V prefix; returns the slot."""
    k, v = synth.kv_prefix(cfg_name, cfg, stream, length, layers=layers, device=gen_device)
    slot = bm.kv_slot_seed(e, k.to("cuda").contiguous(), v.to("cuda").contiguous(), length)
    torch.cuda.synchronize()
    return slot
