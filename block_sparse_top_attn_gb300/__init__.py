"""GB300-native (sm_103a) MSA block-sparse top-k attention backward."""
