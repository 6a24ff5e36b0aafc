"""HSTU attention for GB300 (sm_103a): C-ABI library plus a thin binding."""
