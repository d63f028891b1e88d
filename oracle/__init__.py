"""fp64 CPU oracle of the HiMuon tiled Newton-Schulz map (test infrastructure only).

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package; the product path never does.
"""

from .himuon_oracle import (  # noqa: F401
    DEFAULT_EPS,
    QUINTIC,
    frobenius_normalise,
    full_mac_count,
    full_ns,
    himuon_step,
    momentum,
    ns_mac_count,
    ns_map,
    ns_steps,
    num_tiles,
    quintic_scalar,
    step_coefficients,
    tile_grid,
    tiled_ns,
    tiled_ns_tiles,
    update_scale,
)
