"""GB300 (sm_103a) masked core attention: forward and backward under the
long-context mask families, through the C ABI of liblca_attn.so."""
from .binding import (  # noqa: F401
    EXPORTED,
    PHASES,
    KernelEvents,
    CtaProfile,
    PROFILE_KERNELS,
    launch_count,
    MASK_KINDS,
    LcaError,
    Mask,
    attn_bwd,
    attn_fwd,
    attn_merge,
    cad_plan,
    CadPlan,
    load,
    marshal,
    mask_materialize,
    mask_nnz,
    mask_tile_classes,
    probe_wait_timeout,
    read_status,
    workspace_size,
)


def build(verbose: bool = False) -> str:
    from ._build import build as _b

    return _b(verbose=verbose)
