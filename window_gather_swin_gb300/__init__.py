"""GB300-native block-glue kernels for shifted-window transformers."""
