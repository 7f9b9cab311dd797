"""Shapes and recipes of the synthetic workloads.

Parameter lists follow the architectures the workloads are named after, in
the order a PyTorch module registers them (that order decides the reverse
bucketing walk).  No dataset and no trained weights are involved: every value
comes from the seeded generator (synth.h).

Recipes (all draws are synth_normal / synth_uniform of synth.h):
  replica grads : stream GRAD, step = optimizer step (1-based), replica k,
                  index = buffer (world) index; N(0, grad_sigma^2), encoded in
                  the grad dtype by truncation.
  params        : stream PARAM, step 0, replica 0, index = buffer index;
                  N(0, 0.02^2), truncated to the param dtype; the fp32 master
                  of a bf16/fp16 param holds exactly that truncated value.
  m, v          : zero (optimizer state starts empty), unless a test asks for
                  a warm state (stream EXP_AVG normal, EXP_AVG_SQ uniform).
"""

BF16, F16, F32 = 1, 2, 0


def toy_mlp(dtype=BF16, blocks=4, d_in=512, d_hidden=1024):
    """blocks x {W [d_hidden, d_in], b [d_hidden], W2 [d_in, d_hidden], b2 [d_in]}."""
    ps = []
    for i in range(blocks):
        ps += [dict(name=f"blk{i}.W", numel=d_hidden * d_in, dtype=dtype),
               dict(name=f"blk{i}.b", numel=d_hidden, dtype=dtype),
               dict(name=f"blk{i}.W2", numel=d_in * d_hidden, dtype=dtype),
               dict(name=f"blk{i}.b2", numel=d_in, dtype=dtype)]
    return ps


def gpt2(layers=12, d=768, ffn=3072, vocab=50257, n_pos=1024, dtype=BF16, ln_dtype=F32):
    """GPT-2-shaped: tied embeddings, LayerNorm weight and bias in ln_dtype."""
    ps = [dict(name="wte", numel=vocab * d, dtype=dtype),
          dict(name="wpe", numel=n_pos * d, dtype=dtype)]
    for i in range(layers):
        h = f"h{i}."
        ps += [dict(name=h + "ln_1.weight", numel=d, dtype=ln_dtype),
               dict(name=h + "ln_1.bias", numel=d, dtype=ln_dtype),
               dict(name=h + "attn.c_attn.weight", numel=d * 3 * d, dtype=dtype),
               dict(name=h + "attn.c_attn.bias", numel=3 * d, dtype=dtype),
               dict(name=h + "attn.c_proj.weight", numel=d * d, dtype=dtype),
               dict(name=h + "attn.c_proj.bias", numel=d, dtype=dtype),
               dict(name=h + "ln_2.weight", numel=d, dtype=ln_dtype),
               dict(name=h + "ln_2.bias", numel=d, dtype=ln_dtype),
               dict(name=h + "mlp.c_fc.weight", numel=d * ffn, dtype=dtype),
               dict(name=h + "mlp.c_fc.bias", numel=ffn, dtype=dtype),
               dict(name=h + "mlp.c_proj.weight", numel=ffn * d, dtype=dtype),
               dict(name=h + "mlp.c_proj.bias", numel=d, dtype=dtype)]
    ps += [dict(name="ln_f.weight", numel=d, dtype=ln_dtype),
           dict(name="ln_f.bias", numel=d, dtype=ln_dtype)]
    return ps


def llama(layers, d, ffn, vocab, dtype=BF16, norm_dtype=F32):
    """Llama-shaped: untied embedding / head, SwiGLU MLP, RMSNorm in norm_dtype."""
    ps = [dict(name="embed_tokens", numel=vocab * d, dtype=dtype)]
    for i in range(layers):
        h = f"layers{i}."
        ps += [dict(name=h + "q_proj", numel=d * d, dtype=dtype),
               dict(name=h + "k_proj", numel=d * d, dtype=dtype),
               dict(name=h + "v_proj", numel=d * d, dtype=dtype),
               dict(name=h + "o_proj", numel=d * d, dtype=dtype),
               dict(name=h + "gate_proj", numel=ffn * d, dtype=dtype),
               dict(name=h + "up_proj", numel=ffn * d, dtype=dtype),
               dict(name=h + "down_proj", numel=d * ffn, dtype=dtype),
               dict(name=h + "input_layernorm", numel=d, dtype=norm_dtype),
               dict(name=h + "post_attention_layernorm", numel=d, dtype=norm_dtype)]
    ps += [dict(name="norm", numel=d, dtype=norm_dtype),
           dict(name="lm_head", numel=vocab * d, dtype=dtype)]
    return ps


HP = dict(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _cfg(**kw):
    base = dict(hp=dict(HP), max_norm=1.0, loss_scale=1.0, grad_sigma=1e-3,
                param_sigma=0.02, n_inst=1, average=False, layout="full",
                ranks="all", grad_reduce_in_fp32=True, bucket_size=None,
                pad_for_high_busbw=False, inf_at=None)
    base.update(kw)
    return base


def config(name):
    """The workloads of NAMES, at full size."""
    if name == "toy_mlp_dp4":
        return _cfg(name=name, params=toy_mlp(), dp=4, bucket_size=1_000_000,
                    steps=3, seed=0)
    if name == "gpt2_small_dp8":
        return _cfg(name=name, params=gpt2(), dp=8, bucket_size=40_000_000,
                    steps=3, seed=1, inf_at=dict(step=2, replica=0, buffer_frac=0.5))
    if name == "llama_1p3b_fp16_dp8":
        return _cfg(name=name, params=llama(24, 2048, 5504, 32000, dtype=F16), dp=8,
                    bucket_size=40_000_000, grad_reduce_in_fp32=False,
                    loss_scale=65536.0, grad_sigma=1e-3 * 65536.0, steps=5, seed=2)
    if name == "llama_7b_dp8_rank0":
        return _cfg(name=name, params=llama(32, 4096, 11008, 32000), dp=8,
                    bucket_size=40_000_000, layout="shard", ranks=[0], steps=10, seed=3)
    if name == "llama_7b_dp8_rank0_bf16grads":
        # bf16 replica grads summed in fp32 (grad_reduce_in_fp32 off)
        return _cfg(name=name, params=llama(32, 4096, 11008, 32000), dp=8,
                    bucket_size=40_000_000, grad_reduce_in_fp32=False, layout="shard",
                    ranks=[0], steps=10, seed=3)
    if name == "llama_7b_dp8_rank0_avg":
        # average_in_collective: the replicas are summed, then averaged
        return dict(config("llama_7b_dp8_rank0"), name=name, average=True)
    if name == "llama_7b_dp16_rank0":
        # one instance of 16 ranks: 16 fp32 replica shards of rank 0
        return _cfg(name=name, params=llama(32, 4096, 11008, 32000), dp=16,
                    bucket_size=40_000_000, layout="shard", ranks=[0], steps=10, seed=5)
    if name.startswith("llama_7b_dp16_2x8"):
        bs = {"1m": 1_000_000, "10m": 10_000_000, "40m": 40_000_000,
              "100m": 100_000_000}[name.rsplit("_", 1)[1]]
        return _cfg(name=name, params=llama(32, 4096, 11008, 32000), dp=8, n_inst=2,
                    bucket_size=bs, layout="shard", ranks=[0], steps=10, seed=4)
    raise KeyError(name)


def mini(name):
    """Scaled-down versions of the same workloads, small enough for the
    element-by-element oracle comparison, with ragged parameter sizes."""
    if name == "toy_mlp_dp4":
        return config(name)  # already small: 4.2M params
    if name == "gpt2_small_dp8":
        return _cfg(name=name + "_mini", params=gpt2(layers=2, d=96, ffn=384, vocab=1001,
                                                     n_pos=67),
                    dp=8, bucket_size=40_000, steps=3, seed=11,
                    inf_at=dict(step=2, replica=0, buffer_frac=0.5))
    if name == "llama_1p3b_fp16_dp8":
        return _cfg(name=name + "_mini", params=llama(2, 128, 344, 999, dtype=F16), dp=8,
                    bucket_size=60_000, grad_reduce_in_fp32=False, loss_scale=65536.0,
                    grad_sigma=1e-3 * 65536.0, steps=5, seed=12)
    if name == "llama_7b_dp8_rank0":
        return _cfg(name=name + "_mini", params=llama(3, 256, 688, 1003), dp=8,
                    bucket_size=100_000, layout="shard", ranks=[3], steps=4, seed=13)
    if name.startswith("llama_7b_dp16_2x8"):
        return _cfg(name=name + "_mini", params=llama(3, 256, 688, 1003), dp=8, n_inst=2,
                    bucket_size=20_000, layout="shard", ranks=[5], steps=3, seed=14)
    raise KeyError(name)


NAMES = ["toy_mlp_dp4", "gpt2_small_dp8", "llama_1p3b_fp16_dp8", "llama_7b_dp8_rank0",
         "llama_7b_dp8_rank0_bf16grads", "llama_7b_dp8_rank0_avg", "llama_7b_dp16_rank0",
         "llama_7b_dp16_2x8_1m", "llama_7b_dp16_2x8_10m", "llama_7b_dp16_2x8_40m",
         "llama_7b_dp16_2x8_100m"]
