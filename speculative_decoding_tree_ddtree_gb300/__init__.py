"""DDTree tree-verify step for one GB300 (sm_103a): C-ABI library
(include/lucetree.h, built from csrc/) and its thin Python binding."""
from .lucetree import (  # noqa: F401
    EXPORTED,
    LucetreeError,
    VerifyStep,
    load,
    lucetree_accept,
    lucetree_argmax,
    lucetree_argmax_workspace,
    lucetree_build_anc_mask,
    lucetree_commit,
    lucetree_verify_attn,
    lucetree_verify_attn_workspace,
)
