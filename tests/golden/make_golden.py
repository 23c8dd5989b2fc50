"""Writes the stored oracle results under tests/golden/.

Calls only the oracle and the seeded workload generators. The source pages
print no worked numeric example for this method, so the stored values are
the oracle's own, kept to detect an unintended change to its arithmetic: a
change that moves them must name, in its commit message, the passage of the
pages that justifies it.

Run: python tests/golden/make_golden.py
"""

import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle.paged_attention as orc  # noqa: E402
from paged_kv_gqa_pkv_gb300 import workloads as W  # noqa: E402


def tiny_decode_record():
    c = W.tiny_decode(0)
    bits = W.bf16_bits
    kp, vp, bad = orc.append(bits(c.k_pool), bits(c.v_pool), c.page_table.numpy(),
                             bits(c.k_new), bits(c.v_new), c.batch_idx.numpy(),
                             c.input_pos.numpy(), c.page_size)
    assert not bad
    out, lse, bad = orc.decode_attention(bits(c.q), kp, vp, c.page_table.numpy(),
                                         c.batch_idx.numpy(), c.seq_lens.numpy(),
                                         c.page_size, c.scale)
    assert not bad
    out_bits = orc.f64_to_bf16_bits(out)
    return {
        "workload": "tiny_decode seed 0 (append then decode)",
        "k_pool_sha256": hashlib.sha256(kp.tobytes()).hexdigest(),
        "v_pool_sha256": hashlib.sha256(vp.tobytes()).hexdigest(),
        "out_bf16_sha256": hashlib.sha256(out_bits.tobytes()).hexdigest(),
        "lse": [[float(x).hex() for x in row] for row in lse],
    }


if __name__ == "__main__":
    rec = tiny_decode_record()
    with open(os.path.join(HERE, "tiny_decode_oracle.json"), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    print("wrote tiny_decode_oracle.json")
