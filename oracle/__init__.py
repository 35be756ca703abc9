"""Float64 CPU oracle for causal Local Linear Attention: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of ``bench.py``
may import this package. It shares no code with ``local_linear_attention_gb300``.
"""
from .lla_oracle import (  # noqa: F401
    lla_row,
    lla_forward_oracle,
    lla_moments_oracle,
    softmax_attention_oracle,
)
from .parallax_oracle import (  # noqa: F401
    parallax_row,
    parallax_forward_oracle,
    parallax_backward_row,
    parallax_backward_oracle,
)
