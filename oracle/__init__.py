"""Float64 CPU oracle for paged-KV GQA attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the package
``paged_kv_gqa_pkv_gb300`` and its CUDA library) imports, links or runs this
package. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may call it.

The oracle is written from the source pages' description of the method and
shares no code, constant or helper with the CUDA path. See
``oracle/paged_attention.py`` for what each function computes and which
passage it follows.
"""

from .paged_attention import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    physical_slot,
    append,
    rope,
    append_rope,
    gather_logical,
    attend,
    decode_attention,
    prefill_attention,
)
