"""fp64 CPU oracle of the hybrid GDN + sink/sliding-window softmax layer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may use it; the CUDA library never does.  It shares no code with
the CUDA path.  See ``oracle/hla_oracle.c`` for the passages each function
follows; ``oracle/backward.py`` restates the layer in fp64 PyTorch for its
gradients.
"""
from .oracle import (  # noqa: F401
    OracleCfg,
    build,
    conv,
    gdn_delayed,
    key_stats,
    key_visible,
    l2norm,
    layer_unit,
    layer_units,
    rope,
    window_softmax,
)
