"""CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (``exact_attention_69_gb300``)
never imports it and shares no code with it.

Two independent statements of the same definition live here:

* ``attn_oracle.c`` (loaded through ``ctypes``): fp64, one row at a time,
  OpenMP over rows; used for every parity check.
* ``reference_np.py``: a dense numpy twin that builds the full mask matrix from
  window coordinate sets; used only on tiny shapes to cross-check the C code.

Definition (both): for each (b, h, i) and keys j in the allowed set A(i),
s_ij = scale * q_i . k_j, o_i = sum_j softmax_j(s_ij) v_j, lse_i = ln sum_j
exp(s_ij). Sources: "Fused Self Attention" (NKI tutorial), section
"Background"; "Profiling in PyTorch" part 3, section "Deconstructing Naive
Attention" (scale, masked_fill with -inf, softmax, matmul); NATTEN issue #142
for the neighbourhood windows and the float32 logsumexp output.

The backward pass (``attention_bwd``) gives dq, dk, dv of a loss whose gradient at
the output is dout, by the chain rule through the same definition.
"""
from .oracle import (  # noqa: F401
    MASK_CAUSAL,
    MASK_CODES,
    MASK_NA2D,
    MASK_NONE,
    SOURCE,
    Oracle,
    allowed,
    attention,
    attention_bwd,
    attention_rows,
    build,
    compile_oracle,
    default,
    library_path,
    max_threads,
)
