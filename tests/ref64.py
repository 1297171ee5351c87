"""An independent float64 GPT-2 forward assembled from torch library routines
(layer_norm, scaled_dot_product_attention with a causal mask, tanh gelu,
matmul) on the checkpoint-layout weights: the exact-arithmetic reference the
oracle is pinned to, and the yardstick of the fp32 error on inputs whose
conditioning sets that error (the stress inputs of synth.py)."""
import numpy as np
import torch
import torch.nn.functional as F


def torch_gpt2_logits(cfg, w, tokens, kv_round=None):
    """Float64 GPT-2 forward over a whole sequence, from library routines.
    kv_round="bf16": k and v rounded through fp32 to bf16 (torch's own
    round-to-nearest-even conversion) before the attention, as a bf16 KV
    cache holds them."""
    d = lambda a: torch.from_numpy(np.asarray(a, np.float32)).double()
    E, H, D = cfg.n_embd, cfg.n_head, cfg.head_dim
    t = torch.as_tensor(np.asarray(tokens, np.int64))
    n = t.numel()
    x = d(w["wte"])[t] + d(w["wpe"])[:n]
    for L in w["layers"]:
        h = F.layer_norm(x, (E,), d(L["ln1_w"]), d(L["ln1_b"]), eps=cfg.ln_eps)
        qkv = h @ d(L["attn_w"]) + d(L["attn_b"])
        q, k, v = qkv.split(E, dim=-1)
        if kv_round == "bf16":
            k, v = (a.float().bfloat16().double() for a in (k, v))
        q, k, v = (a.reshape(n, H, D).transpose(0, 1) for a in (q, k, v))
        a = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        a = a.transpose(0, 1).reshape(n, E)
        x = x + a @ d(L["proj_w"]) + d(L["proj_b"])
        h = F.layer_norm(x, (E,), d(L["ln2_w"]), d(L["ln2_b"]), eps=cfg.ln_eps)
        f = F.gelu(h @ d(L["fc_w"]) + d(L["fc_b"]), approximate="tanh")
        x = x + f @ d(L["mlp_proj_w"]) + d(L["mlp_proj_b"])
    x = F.layer_norm(x, (E,), d(w["ln_f_w"]), d(w["ln_f_b"]), eps=cfg.ln_eps)
    head = w.get("head", w["wte"])     # a separately stored head, else the tied wte
    return (x @ d(head).T).numpy()
