"""Entropy report of compressed KV caches.

The method packs the lattice indices at b bits per coordinate, optionally
delta-codes them along tokens and leaves the rest to a general-purpose entropy
coder on the host.  The coder itself is not part of this library; this module
states what an ideal order-0 coder could reach on the codes the GPU produced:
the empirical entropy of the b-bit field symbols (with and without the
temporal delta), of the idx bytes, and of the coset bits, next to the raw
rate of the packed format.  The counts come from nq_code_histogram.

    python -m e8_lattice_vector_gb300.entropy --config mistral7b --layers 4
"""
import argparse
import json
import math

import torch


def entropy_bits(counts):
    """Order-0 empirical entropy in bits per symbol of a count vector."""
    counts = [int(c) for c in counts if int(c) > 0]
    n = sum(counts)
    if n == 0:
        return 0.0
    return 0.0 - sum(c / n * math.log2(c / n) for c in counts)


def summarize(counts, bits, padded_dim, group):
    """Rates in bits per coordinate for one tensor's counters [274]."""
    c = [int(v) for v in counts]
    fields = c[0:16][: 1 << bits]
    nfield = sum(fields)
    blocks = c[272] + c[273]
    h_field = entropy_bits(fields)
    h_byte = entropy_bits(c[16:272])
    h_coset = entropy_bits(c[272:274])
    scale_bits = 16.0 * (padded_dim // group) / padded_dim
    return {
        "fields": nfield,
        "field_entropy_bits": round(h_field, 4),
        "byte_entropy_bits_per_byte": round(h_byte, 4),
        "coset_entropy_bits_per_block": round(h_coset, 4),
        "half_coset_share": round(c[273] / blocks, 4) if blocks else 0.0,
        "raw_bits_per_coord": round(bits + 1.0 / 8 + scale_bits, 4),
        "order0_bits_per_coord": round(h_field + h_coset / 8 + scale_bits, 4),
    }


def report(K, V, params, rope=None):
    """Compress K, V with params and summarize the codes of both tensors."""
    from . import codec

    shape = codec.shape_of(K)
    buf = codec.compress_kv(K, V, params, rope)
    counts = codec.code_histogram(buf, shape, params).cpu()
    lay = codec.plan(shape, params)
    dp = int(lay.padded_dim)
    return {
        "k": summarize(counts[0], params.key_bits, dp, params.group_size),
        "v": summarize(counts[1], params.value_bits, dp, params.group_size),
    }


def main(argv=None):
    from . import codec
    from .synth import CONFIGS, make_cache

    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--config", default="mistral7b", choices=sorted(CONFIGS))
    ap.add_argument("--layers", type=int, default=None, help="first N layers only")
    ap.add_argument("--delta-chunk", type=int, default=256, help="delta restart interval for the delta row")
    a = ap.parse_args(argv)
    cfg = CONFIGS[a.config]
    K, V = make_cache(cfg, device="cuda", layers=a.layers)
    for params in cfg.modes:
        rope = codec.RopeTable.build(cfg.tokens, cfg.head_dim, params.rope_theta) if params.rope_theta > 0 else None
        for delta in (0, a.delta_chunk):
            p = codec.CodecParams(params.key_bits, params.value_bits, params.group_size, params.strict, delta,
                                  params.rope_theta)
            rec = {"config": cfg.name, "layers": int(K.shape[0]), "key_bits": p.key_bits, "value_bits": p.value_bits,
                   "group": p.group_size, "strict": bool(p.strict), "delta_chunk": delta}
            rec.update(report(K, V, p, rope))
            print(json.dumps(rec), flush=True)
    torch.cuda.synchronize()


if __name__ == "__main__":
    main()
